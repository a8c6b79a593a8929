// Host block allocator of the paged KV cache.
//
// Sources: foundry page on paged block allocation ("In and out": a free pool
// that is a stack of physical indices; blocks taken on demand, one per
// block_size tokens, appended to the sequence's block table; a reference
// count raised when a block is shared; "Concept": fork copies the table, not
// the memory, and a block is copied only when a branch writes into it);
// "PagedAttention, clearly explained" (a block is assigned only when the
// previous one fills; finished requests return their blocks at once);
// "PagedAttention Memory Management", "Complex Topologies and Memory Sharing"
// (the shared prompt blocks' count equals the number of sequences mapping
// them).
//
// Every mutating call first works out how many blocks it will pop and fails
// before touching anything when the stack is short, so calls are
// all-or-nothing.  A batch append keeps an undo record per sequence and rolls
// back in reverse order when a later sequence fails, which restores the
// stack order exactly (pops and pushes are mirror images).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <limits>
#include <new>
#include <unordered_map>
#include <vector>

#include "common.h"

namespace pkv {

namespace {
thread_local std::string g_last_error;
}

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

struct Seq {
  std::vector<int32_t> table;  // logical block -> physical block
  int64_t len = 0;             // tokens written (slots reserved)
};

// What one single-sequence append changed, enough to undo it.
struct AppendUndo {
  int64_t seq_id;
  int64_t old_len;
  size_t old_table_size;
  bool cow;
  int32_t cow_index;
  int32_t cow_src;
};

}  // namespace pkv

struct pkv_pool {
  int32_t num_blocks;
  int32_t block_size;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, pkv::Seq> seqs;
};

namespace pkv {
namespace {

inline int64_t blocks_for(int64_t tokens, int32_t t) { return (tokens + t - 1) / t; }

// Blocks an append of n_new tokens pops, and whether its first token lands in
// a shared, partly filled block (copy-on-write).
int64_t blocks_needed(const pkv_pool* p, const Seq& s, int64_t n_new, bool* cow) {
  const int32_t t = p->block_size;
  *cow = n_new > 0 && s.len % t != 0 && p->refcount[s.table[s.len / t]] > 1;
  const int64_t opened = blocks_for(s.len + n_new, t) - blocks_for(s.len, t);
  return opened + (*cow ? 1 : 0);
}

pkv_status append_one(pkv_pool* p, int64_t seq_id, Seq& s, int64_t n_new, int64_t* slots_out,
                      int32_t* cow_out, int32_t cow_cap, int32_t* n_cow, AppendUndo* undo) {
  bool cow = false;
  const int64_t need = blocks_needed(p, s, n_new, &cow);
  if (need > static_cast<int64_t>(p->free_stack.size())) {
    set_error("sequence %lld needs %lld blocks, %zu free", (long long)seq_id, (long long)need,
              p->free_stack.size());
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  if (cow && (cow_out == nullptr || *n_cow >= cow_cap)) {
    set_error("sequence %lld needs a copy-on-write pair but cow_cap is exhausted",
              (long long)seq_id);
    return PKV_ERR_INVALID_ARG;
  }
  const int32_t t = p->block_size;
  if (undo) {
    undo->seq_id = seq_id;
    undo->old_len = s.len;
    undo->old_table_size = s.table.size();
    undo->cow = cow;
    undo->cow_index = cow ? static_cast<int32_t>(s.len / t) : -1;
    undo->cow_src = cow ? s.table[s.len / t] : -1;
  }
  const int64_t start = s.len;
  for (int64_t pos = start; pos < start + n_new; ++pos) {
    if (pos % t == 0) {
      const int32_t b = p->free_stack.back();
      p->free_stack.pop_back();
      p->refcount[b] = 1;
      s.table.push_back(b);
    } else if (pos == start && cow) {
      const int32_t src = s.table[pos / t];
      const int32_t dst = p->free_stack.back();
      p->free_stack.pop_back();
      p->refcount[dst] = 1;
      p->refcount[src] -= 1;
      s.table[pos / t] = dst;
      cow_out[2 * (*n_cow)] = src;
      cow_out[2 * (*n_cow) + 1] = dst;
      ++(*n_cow);
    }
    if (slots_out) slots_out[pos - start] = static_cast<int64_t>(s.table[pos / t]) * t + pos % t;
  }
  s.len = start + n_new;
  return PKV_OK;
}

// Reverse one append: return its new blocks (last popped first) and its
// copy-on-write block, then restore the shared source.
void undo_append(pkv_pool* p, const AppendUndo& u) {
  Seq& s = p->seqs.at(u.seq_id);
  while (s.table.size() > u.old_table_size) {
    const int32_t b = s.table.back();
    s.table.pop_back();
    p->refcount[b] = 0;
    p->free_stack.push_back(b);
  }
  if (u.cow) {
    const int32_t dst = s.table[u.cow_index];
    p->refcount[dst] = 0;
    p->free_stack.push_back(dst);
    s.table[u.cow_index] = u.cow_src;
    p->refcount[u.cow_src] += 1;
  }
  s.len = u.old_len;
}

}  // namespace
}  // namespace pkv

using pkv::fail;

extern "C" {

uint64_t pkv_block_bytes(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t elem_bytes) {
  if (num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || elem_bytes <= 0)
    return 0;
  return 2ull * (uint64_t)num_layers * (uint64_t)num_kv_heads * (uint64_t)head_dim *
         (uint64_t)block_size * (uint64_t)elem_bytes;
}

uint64_t pkv_num_blocks_for_budget(uint64_t budget_bytes, uint64_t block_bytes) {
  return block_bytes == 0 ? 0 : budget_bytes / block_bytes;
}

int32_t pkv_dtype_bytes(int32_t dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_E4M3: return 1;
    default: return 0;
  }
}

pkv_status pkv_pool_create(int32_t num_blocks, int32_t block_size,
                           const int32_t* initial_free_order, pkv_pool** out) {
  if (out == nullptr) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks and block_size must be positive");
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->refcount.assign(num_blocks, 0);
  p->free_stack.resize(num_blocks);
  if (initial_free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = initial_free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete p;
        return fail(PKV_ERR_INVALID_ARG, "initial_free_order is not a permutation of the pool");
      }
      seen[b] = 1;
      p->free_stack[num_blocks - 1 - i] = b;
    }
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) p->free_stack[num_blocks - 1 - i] = i;
  }
  *out = p;
  return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

pkv_status pkv_seq_create(pkv_pool* pool, int64_t seq_id) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (pool->seqs.count(seq_id)) {
    pkv::set_error("sequence %lld exists", (long long)seq_id);
    return PKV_ERR_INVALID_ARG;
  }
  pool->seqs.emplace(seq_id, pkv::Seq{});
  return PKV_OK;
}

pkv_status pkv_seq_append(pkv_pool* pool, int64_t seq_id, int32_t n_new, int64_t* slots_out,
                          int32_t* cow_out, int32_t cow_cap, int32_t* n_cow_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_new < 0) return fail(PKV_ERR_INVALID_ARG, "n_new is negative");
  if (n_new > 0 && !slots_out) return fail(PKV_ERR_INVALID_ARG, "slots_out is NULL");
  if (cow_cap < 0) return fail(PKV_ERR_INVALID_ARG, "cow_cap is negative");
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)seq_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  int32_t n_cow = 0;
  const pkv_status st =
      pkv::append_one(pool, seq_id, it->second, n_new, slots_out, cow_out, cow_cap, &n_cow, nullptr);
  if (n_cow_out) *n_cow_out = (st == PKV_OK) ? n_cow : 0;
  return st;
}

pkv_status pkv_batch_append(pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                            int64_t* slots_out, int32_t* cow_out, int32_t cow_cap,
                            int32_t* n_cow_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "n_seqs is negative");
  if (n_seqs > 0 && (!seq_ids || !slots_out))
    return fail(PKV_ERR_INVALID_ARG, "seq_ids or slots_out is NULL");
  if (cow_cap < 0) return fail(PKV_ERR_INVALID_ARG, "cow_cap is negative");
  std::vector<pkv::AppendUndo> undo;
  undo.reserve(n_seqs);
  int32_t n_cow = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = pool->seqs.find(seq_ids[i]);
    pkv_status st;
    if (it == pool->seqs.end()) {
      pkv::set_error("unknown sequence %lld", (long long)seq_ids[i]);
      st = PKV_ERR_UNKNOWN_SEQ;
    } else {
      undo.emplace_back();
      st = pkv::append_one(pool, seq_ids[i], it->second, 1, slots_out + i, cow_out, cow_cap,
                           &n_cow, &undo.back());
      if (st != PKV_OK) undo.pop_back();
    }
    if (st != PKV_OK) {
      for (auto u = undo.rbegin(); u != undo.rend(); ++u) pkv::undo_append(pool, *u);
      if (n_cow_out) *n_cow_out = 0;
      return st;
    }
  }
  if (n_cow_out) *n_cow_out = n_cow;
  return PKV_OK;
}

pkv_status pkv_seq_fork(pkv_pool* pool, int64_t parent_id, int64_t child_id) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  auto it = pool->seqs.find(parent_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)parent_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  if (pool->seqs.count(child_id)) {
    pkv::set_error("sequence %lld exists", (long long)child_id);
    return PKV_ERR_INVALID_ARG;
  }
  pkv::Seq child = it->second;  // copy the table, not the memory
  for (int32_t b : child.table) pool->refcount[b] += 1;
  pool->seqs.emplace(child_id, std::move(child));
  return PKV_OK;
}

pkv_status pkv_seq_free(pkv_pool* pool, int64_t seq_id) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)seq_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  for (int32_t b : it->second.table) {
    if (--pool->refcount[b] == 0) pool->free_stack.push_back(b);
  }
  pool->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_seq_table(const pkv_pool* pool, int64_t seq_id, int32_t* out, int32_t cap,
                         int32_t* n_blocks, int64_t* context_len) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)seq_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  const auto& tab = it->second.table;
  if (cap > 0 && !out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  if (cap > 0 && cap < static_cast<int32_t>(tab.size()))
    return fail(PKV_ERR_INVALID_ARG, "cap is smaller than the table");
  if (cap > 0) std::copy(tab.begin(), tab.end(), out);
  if (n_blocks) *n_blocks = static_cast<int32_t>(tab.size());
  if (context_len) *context_len = it->second.len;
  return PKV_OK;
}

pkv_status pkv_block_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                            int32_t max_blocks, int32_t* tables_out, int32_t* context_lens_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_seqs < 0 || max_blocks < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n_seqs > 0 && (!seq_ids || !tables_out || !context_lens_out))
    return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  // validate first so a failure leaves the outputs untouched
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = pool->seqs.find(seq_ids[i]);
    if (it == pool->seqs.end()) {
      pkv::set_error("unknown sequence %lld", (long long)seq_ids[i]);
      return PKV_ERR_UNKNOWN_SEQ;
    }
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks)
      return fail(PKV_ERR_INVALID_ARG, "a block table is longer than max_blocks");
    if (it->second.len > std::numeric_limits<int32_t>::max())
      return fail(PKV_ERR_INVALID_ARG, "a context length exceeds INT32_MAX");
  }
  for (int32_t i = 0; i < n_seqs; ++i) {
    const auto& s = pool->seqs.find(seq_ids[i])->second;
    int32_t* row = tables_out + static_cast<int64_t>(i) * max_blocks;
    const int32_t n = static_cast<int32_t>(s.table.size());
    std::copy(s.table.begin(), s.table.end(), row);
    std::fill(row + n, row + max_blocks, -1);
    context_lens_out[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

pkv_status pkv_block_refcount(const pkv_pool* pool, int32_t block, int32_t* refcount) {
  if (!pool || !refcount) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  if (block < 0 || block >= pool->num_blocks) return fail(PKV_ERR_INVALID_ARG, "block out of range");
  *refcount = pool->refcount[block];
  return PKV_OK;
}

int32_t pkv_num_free_blocks(const pkv_pool* pool) {
  return pool ? static_cast<int32_t>(pool->free_stack.size()) : 0;
}

pkv_status pkv_free_stack(const pkv_pool* pool, int32_t* out, int32_t cap, int32_t* n) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  const int32_t sz = static_cast<int32_t>(pool->free_stack.size());
  if (cap > 0 && !out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  if (cap > 0 && cap < sz) return fail(PKV_ERR_INVALID_ARG, "cap is smaller than the stack");
  if (cap > 0) std::copy(pool->free_stack.rbegin(), pool->free_stack.rend(), out);
  if (n) *n = sz;
  return PKV_OK;
}

pkv_status pkv_pool_usage(const pkv_pool* pool, int64_t* live_seqs, int64_t* live_tokens,
                          int64_t* used_blocks) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  int64_t tokens = 0;
  for (const auto& kv : pool->seqs) tokens += kv.second.len;
  if (live_seqs) *live_seqs = static_cast<int64_t>(pool->seqs.size());
  if (live_tokens) *live_tokens = tokens;
  if (used_blocks) *used_blocks = pool->num_blocks - static_cast<int64_t>(pool->free_stack.size());
  return PKV_OK;
}

}  // extern "C"

extern "C" const char* pkv_last_error(void) { return pkv::g_last_error.c_str(); }
