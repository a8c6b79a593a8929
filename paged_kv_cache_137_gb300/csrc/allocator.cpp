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
// Prefix caching (foundry page, "The knobs": enable_prefix_caching hashes each
// filled block so that unrelated requests share physical blocks; "Failure
// modes": sharing is block-granular; katajob Q&A, "Sharing, the second
// dividend": if the tokens match, the blocks holding their KV state are reused
// and that part of prefill is skipped) is optional per pool.  A full block is
// published under the exact key (entry of the previous block, its T token
// ids); a new sequence created from a prompt takes the longest chain of
// published blocks that matches its first tokens, keeping at least one prompt
// token to compute.  A published block whose count drops to zero is kept, in
// least-recently-freed order, and handed out again only when the free stack
// is empty (eviction: the oldest first, a sequence's last block before its
// first).
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
#include <list>
#include <new>
#include <string>
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
  // prefix caching: token ids of positions 0 .. len - 1 while they are known
  // (tokens.size() == len), and per full block the cache entry of its content
  // (-1: not published / unknown)
  std::vector<int32_t> tokens;
  std::vector<int64_t> chain;
  // unique over the pool's life: a new sequence (also a fork child, or an id
  // used again) gets a new one, so a caller's copy of a table can tell
  int64_t incarnation = 0;
  // batch-append check only: tokens of the batch already counted for this
  // sequence (0 outside the check)
  int32_t pending = 0;
};

// One published block and its content key bytes (parent entry, token ids).
struct CacheEntry {
  std::string key;
  int32_t block;
};

// What one single-sequence append changed, enough to undo it.
struct AppendUndo {
  int64_t seq_id;
  int64_t old_len;
  size_t old_table_size;
  size_t old_chain_size;
  size_t old_tokens_size;
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
  // batch-append check only: counts the batch's earlier copies take from a
  // block (0 outside the check)
  std::vector<int32_t> rc_taken;
  std::unordered_map<int64_t, pkv::Seq> seqs;
  // prefix cache (off unless enabled)
  bool caching = false;
  int64_t next_entry = 1;                                 // entry 0 is the root (no parent)
  std::unordered_map<std::string, int64_t> key_to_entry;  // key bytes -> entry
  std::unordered_map<int64_t, pkv::CacheEntry> entries;   // entry -> key, block
  std::vector<int64_t> block_entry;                       // block -> entry, -1 if none
  std::list<int32_t> lru;                                 // cached blocks at count 0, oldest first
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<char> in_lru;
  int64_t hit_tokens = 0, evictions = 0;
  int64_t next_incarnation = 1;  // 0 never names a sequence
};

namespace pkv {
namespace {

inline int64_t blocks_for(int64_t tokens, int32_t t) { return (tokens + t - 1) / t; }

// Insert a new sequence under a fresh incarnation number.
Seq& add_seq(pkv_pool* p, int64_t seq_id, Seq&& s) {
  s.incarnation = p->next_incarnation++;
  return p->seqs.emplace(seq_id, std::move(s)).first->second;
}

// Blocks a pop can hand out: the free stack, then (with prefix caching) the
// cached blocks nobody references.
inline int64_t available(const pkv_pool* p) {
  return static_cast<int64_t>(p->free_stack.size()) + static_cast<int64_t>(p->lru.size());
}

std::string cache_key(int64_t parent, const int32_t* tokens, int32_t t) {
  std::string k(sizeof(int64_t) + sizeof(int32_t) * t, '\0');
  std::memcpy(&k[0], &parent, sizeof(int64_t));
  std::memcpy(&k[sizeof(int64_t)], tokens, sizeof(int32_t) * t);
  return k;
}

void unpublish(pkv_pool* p, int32_t b) {
  const int64_t e = p->block_entry[b];
  if (e < 0) return;
  auto it = p->entries.find(e);
  if (it != p->entries.end()) {
    p->key_to_entry.erase(it->second.key);
    p->entries.erase(it);
  }
  p->block_entry[b] = -1;
}

// Take a block: the top of the free stack, else evict the least recently
// freed cached block (its entry is dropped).  The caller checked available().
int32_t pop_block(pkv_pool* p) {
  if (!p->free_stack.empty()) {
    const int32_t b = p->free_stack.back();
    p->free_stack.pop_back();
    return b;
  }
  const int32_t b = p->lru.front();
  p->lru.pop_front();
  p->in_lru[b] = 0;
  unpublish(p, b);
  ++p->evictions;
  return b;
}

// A block whose count reached zero: kept for reuse if it is published, else
// back on the free stack.
void release_block(pkv_pool* p, int32_t b) {
  if (p->caching && p->block_entry[b] >= 0) {
    p->lru.push_back(b);
    p->lru_pos[b] = std::prev(p->lru.end());
    p->in_lru[b] = 1;
  } else {
    p->free_stack.push_back(b);
  }
}

// A cached block taken by a lookup: out of the reuse list if it was there.
void acquire_cached(pkv_pool* p, int32_t b) {
  if (p->in_lru[b]) {
    p->lru.erase(p->lru_pos[b]);
    p->in_lru[b] = 0;
  }
  p->refcount[b] += 1;
}

// Publish the blocks of s filled by positions [old_len, s.len) (token ids
// known): each gets the entry of an equal published block or a new one.
void publish_filled(pkv_pool* p, pkv::Seq& s, int64_t old_len) {
  const int32_t t = p->block_size;
  (void)old_len;
  for (int64_t i = static_cast<int64_t>(s.chain.size()); (i + 1) * t <= s.len; ++i) {
    const int64_t parent = i == 0 ? 0 : s.chain[i - 1];
    if (parent < 0 || static_cast<int64_t>(s.tokens.size()) < (i + 1) * t) {
      s.chain.push_back(-1);
      continue;
    }
    const std::string key = cache_key(parent, &s.tokens[i * t], t);
    auto it = p->key_to_entry.find(key);
    if (it != p->key_to_entry.end()) {
      s.chain.push_back(it->second);  // equal content already published elsewhere
      continue;
    }
    const int32_t b = s.table[i];
    if (p->block_entry[b] >= 0) {  // shared with a fork sibling that published it
      s.chain.push_back(p->block_entry[b]);
      continue;
    }
    const int64_t e = p->next_entry++;
    p->key_to_entry.emplace(key, e);
    p->entries.emplace(e, CacheEntry{key, b});
    p->block_entry[b] = e;
    s.chain.push_back(e);
  }
}

// Blocks an append of n_new tokens pops, and whether its first token lands in
// a shared, partly filled block (copy-on-write).
int64_t blocks_needed(const pkv_pool* p, const Seq& s, int64_t n_new, bool* cow) {
  const int32_t t = p->block_size;
  *cow = n_new > 0 && s.len % t != 0 && p->refcount[s.table[s.len / t]] > 1;
  const int64_t opened = blocks_for(s.len + n_new, t) - blocks_for(s.len, t);
  return opened + (*cow ? 1 : 0);
}

pkv_status append_one(pkv_pool* p, int64_t seq_id, Seq& s, int64_t n_new, int64_t* slots_out,
                      int32_t* cow_out, int32_t cow_cap, int32_t* n_cow, AppendUndo* undo,
                      const int32_t* token_ids = nullptr) {
  bool cow = false;
  const int64_t need = blocks_needed(p, s, n_new, &cow);
  if (need > available(p)) {
    set_error("sequence %lld needs %lld blocks, %lld free", (long long)seq_id, (long long)need,
              (long long)available(p));
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
    undo->old_chain_size = s.chain.size();
    undo->old_tokens_size = s.tokens.size();
    undo->cow = cow;
    undo->cow_index = cow ? static_cast<int32_t>(s.len / t) : -1;
    undo->cow_src = cow ? s.table[s.len / t] : -1;
  }
  const int64_t start = s.len;
  for (int64_t pos = start; pos < start + n_new; ++pos) {
    if (pos % t == 0) {
      const int32_t b = pop_block(p);
      p->refcount[b] = 1;
      s.table.push_back(b);
    } else if (pos == start && cow) {
      const int32_t src = s.table[pos / t];
      const int32_t dst = pop_block(p);
      p->refcount[dst] = 1;
      p->refcount[src] -= 1;
      s.table[pos / t] = dst;
      cow_out[2 * (*n_cow)] = src;
      cow_out[2 * (*n_cow) + 1] = dst;
      ++(*n_cow);
    }
    if (slots_out) slots_out[pos - start] = static_cast<int64_t>(s.table[pos / t]) * t + pos % t;
  }
  // token ids are kept only while every earlier position's id is known
  if (p->caching) {
    if (token_ids && static_cast<int64_t>(s.tokens.size()) == start)
      s.tokens.insert(s.tokens.end(), token_ids, token_ids + n_new);
  }
  s.len = start + n_new;
  if (p->caching) publish_filled(p, s, start);
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
    if (p->caching) unpublish(p, b);  // published by the undone append
    p->free_stack.push_back(b);
  }
  s.chain.resize(std::min(s.chain.size(), u.old_chain_size));
  s.tokens.resize(std::min(s.tokens.size(), u.old_tokens_size));
  if (u.cow) {
    const int32_t dst = s.table[u.cow_index];
    p->refcount[dst] = 0;
    p->free_stack.push_back(dst);
    s.table[u.cow_index] = u.cow_src;
    p->refcount[u.cow_src] += 1;
  }
  s.len = u.old_len;
}

// Finish a sequence: its blocks whose count reaches zero go back on the stack
// in logical order (published ones are kept for reuse, last block first, so
// that a sequence's tail is evicted before its prefix).
void free_seq_blocks(pkv_pool* pool, std::unordered_map<int64_t, pkv::Seq>::iterator it) {
  const auto& tab = it->second.table;
  if (pool->caching) {
    for (auto b = tab.rbegin(); b != tab.rend(); ++b)
      if (pool->block_entry[*b] >= 0 && --pool->refcount[*b] == 0) release_block(pool, *b);
    for (int32_t b : tab)
      if (pool->block_entry[b] < 0 && --pool->refcount[b] == 0) pool->free_stack.push_back(b);
  } else {
    for (int32_t b : tab)
      if (--pool->refcount[b] == 0) pool->free_stack.push_back(b);
  }
  pool->seqs.erase(it);
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
  pkv::add_seq(pool, seq_id, pkv::Seq{});
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
  // check the whole batch first, so that a short pool changes nothing (and
  // no cached block is evicted for a batch that then fails)
  // (in batch order, with running totals, so that the first failing
  // sequence and its error are the ones a sequential append would meet)
  // the sequences found here serve the second pass too (appends insert no
  // sequence, so the pointers stay valid); both buffers are reused per thread
  static thread_local std::vector<pkv::Seq*> batch;
  static thread_local std::vector<pkv::AppendUndo> undo;
  batch.clear();
  undo.clear();
  // The check follows the sequential appends exactly: a sequence named k
  // times takes tokens len .. len + k - 1, each counted at its own position,
  // and only its first can need a copy (the block it then writes is its
  // own); a copy takes one count from its source block, so a later sharer
  // of that block may find it private and write in place.
  static thread_local std::vector<int32_t> taken;  // blocks with a count taken
  taken.clear();
  if (pool->rc_taken.size() != pool->refcount.size()) pool->rc_taken.assign(pool->refcount.size(), 0);
  {
    pkv_status st = PKV_OK;
    int64_t need = 0, cows = 0;
    const int32_t t = pool->block_size;
    for (int32_t i = 0; i < n_seqs && st == PKV_OK; ++i) {
      auto it = pool->seqs.find(seq_ids[i]);
      if (it == pool->seqs.end()) {
        pkv::set_error("unknown sequence %lld", (long long)seq_ids[i]);
        st = PKV_ERR_UNKNOWN_SEQ;
        break;
      }
      pkv::Seq& s = it->second;
      batch.push_back(&s);
      const int64_t k = s.pending++;
      const int64_t pos = s.len + k;
      bool cow = false;
      if (pos % t == 0) {
        need += 1;  // opens a block
      } else if (k == 0) {
        const int32_t b = s.table[pos / t];
        cow = pool->refcount[b] - pool->rc_taken[b] > 1;
        if (cow) {
          need += 1;
          if (pool->rc_taken[b]++ == 0) taken.push_back(b);
        }
      }
      if (need > pkv::available(pool)) {
        pkv::set_error("sequence %lld: the batch needs %lld blocks, %lld free",
                       (long long)seq_ids[i], (long long)need, (long long)pkv::available(pool));
        st = PKV_ERR_OUT_OF_BLOCKS;
      } else if (cow && (cow_out == nullptr || ++cows > cow_cap)) {
        pkv::set_error("sequence %lld needs a copy-on-write pair but cow_cap is exhausted",
                       (long long)seq_ids[i]);
        st = PKV_ERR_INVALID_ARG;
      }
    }
    for (pkv::Seq* s : batch) s->pending = 0;
    for (int32_t b : taken) pool->rc_taken[b] = 0;
    if (st != PKV_OK) return st;
  }
  // The check above is exact, so no append below fails; the undo records
  // are a safety net that would restore the state if one did.
  int32_t n_cow = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    undo.emplace_back();
    const pkv_status st = pkv::append_one(pool, seq_ids[i], *batch[i], 1, slots_out + i, cow_out,
                                          cow_cap, &n_cow, &undo.back());
    if (st != PKV_OK) {
      undo.pop_back();
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
  pkv::add_seq(pool, child_id, std::move(child));
  return PKV_OK;
}

pkv_status pkv_seq_free(pkv_pool* pool, int64_t seq_id) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)seq_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  pkv::free_seq_blocks(pool, it);
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

pkv_status pkv_block_tables_update(const pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                                   int32_t max_blocks, int32_t* tables_inout, int64_t* rows_inout,
                                   int32_t* context_lens_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_seqs < 0 || max_blocks < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n_seqs > 0 && (!seq_ids || !tables_inout || !rows_inout || !context_lens_out))
    return fail(PKV_ERR_INVALID_ARG, "NULL argument");
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
    int32_t* row = tables_inout + static_cast<int64_t>(i) * max_blocks;
    int64_t* state = rows_inout + 2 * static_cast<int64_t>(i);
    const int64_t n = static_cast<int64_t>(s.table.size());
    // Between two calls a live sequence's table only grows at its end, and
    // a copy-on-write replaces the entry at len / T, which is at least the
    // last entry the row held (len never shrinks).  So a row last written
    // for this incarnation is rewritten from its last entry on; any other
    // row is written whole.
    // state: the incarnation, then (max_blocks << 32) | entries held
    const int64_t held = state[1] & 0xffffffffLL;
    int64_t from = 0;
    if (state[0] == s.incarnation && (state[1] >> 32) == max_blocks && held <= n) {
      from = std::max<int64_t>(held - 1, 0);
    } else {
      std::fill(row + n, row + max_blocks, -1);
    }
    std::copy(s.table.begin() + from, s.table.end(), row + from);
    state[0] = s.incarnation;
    state[1] = (static_cast<int64_t>(max_blocks) << 32) | n;
    context_lens_out[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

pkv_status pkv_shared_prefix_blocks(const pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                                    int32_t* n_blocks) {
  if (!pool || !n_blocks) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  if (n_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n_seqs > 0 && !seq_ids) return fail(PKV_ERR_INVALID_ARG, "seq_ids is NULL");
  std::vector<const pkv::Seq*> seqs(static_cast<size_t>(n_seqs));
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = pool->seqs.find(seq_ids[i]);
    if (it == pool->seqs.end()) {
      pkv::set_error("unknown sequence %lld", (long long)seq_ids[i]);
      return PKV_ERR_UNKNOWN_SEQ;
    }
    seqs[i] = &it->second;
  }
  int64_t k = 0;
  if (n_seqs > 0) {
    // full blocks before every sequence's last position
    k = std::numeric_limits<int64_t>::max();
    for (const pkv::Seq* s : seqs) k = std::min<int64_t>(k, s->len > 0 ? (s->len - 1) / pool->block_size : 0);
    const std::vector<int32_t>& t0 = seqs[0]->table;
    for (const pkv::Seq* s : seqs) {
      int64_t i = 0;
      while (i < k && s->table[i] == t0[i]) ++i;
      k = i;
    }
  }
  *n_blocks = static_cast<int32_t>(std::min<int64_t>(k, std::numeric_limits<int32_t>::max()));
  return PKV_OK;
}

pkv_status pkv_block_refcount(const pkv_pool* pool, int32_t block, int32_t* refcount) {
  if (!pool || !refcount) return fail(PKV_ERR_INVALID_ARG, "NULL argument");
  if (block < 0 || block >= pool->num_blocks) return fail(PKV_ERR_INVALID_ARG, "block out of range");
  *refcount = pool->refcount[block];
  return PKV_OK;
}

int32_t pkv_num_free_blocks(const pkv_pool* pool) {
  return pool ? static_cast<int32_t>(pkv::available(pool)) : 0;
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
  if (used_blocks) *used_blocks = pool->num_blocks - pkv::available(pool);
  return PKV_OK;
}

pkv_status pkv_pool_enable_prefix_cache(pkv_pool* pool) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (pool->caching) return PKV_OK;
  if (!pool->seqs.empty()) return fail(PKV_ERR_INVALID_ARG, "enable prefix caching before any sequence");
  pool->caching = true;
  pool->block_entry.assign(pool->num_blocks, -1);
  pool->lru_pos.resize(pool->num_blocks);
  pool->in_lru.assign(pool->num_blocks, 0);
  return PKV_OK;
}

pkv_status pkv_seq_create_cached(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                                 int32_t n_tokens, int32_t* n_cached) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (!pool->caching) return fail(PKV_ERR_INVALID_ARG, "prefix caching is not enabled");
  if (n_tokens < 0 || (n_tokens > 0 && !token_ids)) return fail(PKV_ERR_INVALID_ARG, "bad token ids");
  if (pool->seqs.count(seq_id)) {
    pkv::set_error("sequence %lld exists", (long long)seq_id);
    return PKV_ERR_INVALID_ARG;
  }
  pkv::Seq s;
  const int32_t t = pool->block_size;
  // the longest chain of published blocks matching the prompt's first full
  // blocks, leaving at least one prompt token to compute
  const int64_t max_blocks = n_tokens > 0 ? (static_cast<int64_t>(n_tokens) - 1) / t : 0;
  for (int64_t i = 0; i < max_blocks; ++i) {
    const int64_t parent = i == 0 ? 0 : s.chain.back();
    auto it = pool->key_to_entry.find(pkv::cache_key(parent, token_ids + i * t, t));
    if (it == pool->key_to_entry.end()) break;
    const int32_t b = pool->entries.at(it->second).block;
    pkv::acquire_cached(pool, b);
    s.table.push_back(b);
    s.chain.push_back(it->second);
  }
  s.len = static_cast<int64_t>(s.table.size()) * t;
  s.tokens.assign(token_ids, token_ids + s.len);
  pool->hit_tokens += s.len;
  if (n_cached) *n_cached = static_cast<int32_t>(s.len);
  pkv::add_seq(pool, seq_id, std::move(s));
  return PKV_OK;
}

pkv_status pkv_seq_append_tokens(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                                 int32_t n_new, int64_t* slots_out, int32_t* cow_out,
                                 int32_t cow_cap, int32_t* n_cow_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_new < 0) return fail(PKV_ERR_INVALID_ARG, "n_new is negative");
  if (n_new > 0 && (!slots_out || !token_ids))
    return fail(PKV_ERR_INVALID_ARG, "slots_out or token_ids is NULL");
  if (cow_cap < 0) return fail(PKV_ERR_INVALID_ARG, "cow_cap is negative");
  auto it = pool->seqs.find(seq_id);
  if (it == pool->seqs.end()) {
    pkv::set_error("unknown sequence %lld", (long long)seq_id);
    return PKV_ERR_UNKNOWN_SEQ;
  }
  int32_t n_cow = 0;
  const pkv_status st = pkv::append_one(pool, seq_id, it->second, n_new, slots_out, cow_out,
                                        cow_cap, &n_cow, nullptr, token_ids);
  if (n_cow_out) *n_cow_out = (st == PKV_OK) ? n_cow : 0;
  return st;
}

pkv_status pkv_prefix_cache_stats(const pkv_pool* pool, int64_t* published_blocks,
                                  int64_t* reusable_blocks, int64_t* hit_tokens,
                                  int64_t* evictions) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (published_blocks) *published_blocks = static_cast<int64_t>(pool->entries.size());
  if (reusable_blocks) *reusable_blocks = static_cast<int64_t>(pool->lru.size());
  if (hit_tokens) *hit_tokens = pool->hit_tokens;
  if (evictions) *evictions = pool->evictions;
  return PKV_OK;
}

pkv_status pkv_reusable_blocks(const pkv_pool* pool, int32_t* out, int32_t cap, int32_t* n) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  const int32_t sz = static_cast<int32_t>(pool->lru.size());
  if (cap > 0 && !out) return fail(PKV_ERR_INVALID_ARG, "out is NULL");
  if (cap > 0 && cap < sz) return fail(PKV_ERR_INVALID_ARG, "cap is smaller than the list");
  if (cap > 0) std::copy(pool->lru.begin(), pool->lru.end(), out);
  if (n) *n = sz;
  return PKV_OK;
}

// ------------------------------------------------------------- preemption
// Foundry page, "The knobs" and "Effect": when the pool cannot satisfy a
// running sequence the engine preempts it, drops its blocks and re-prefills
// it later (recompute), instead of failing; "Failure modes": a free-block
// watermark keeps admissions from driving the pool into constant preemption.


pkv_status pkv_batch_append_preempt(pkv_pool* pool, const int64_t* seq_ids, int32_t n_seqs,
                                    int64_t* slots_out, int32_t* cow_out, int32_t cow_cap,
                                    int32_t* n_cow_out, int64_t* preempted_out,
                                    int32_t* n_preempted_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "n_seqs is negative");
  if (n_seqs > 0 && (!seq_ids || !slots_out || !preempted_out))
    return fail(PKV_ERR_INVALID_ARG, "seq_ids, slots_out or preempted_out is NULL");
  if (cow_cap < n_seqs || (n_seqs > 0 && !cow_out))
    return fail(PKV_ERR_INVALID_ARG, "cow_out must hold n_seqs pairs");
  {
    std::unordered_map<int64_t, int> seen;
    for (int32_t i = 0; i < n_seqs; ++i) {
      if (!pool->seqs.count(seq_ids[i])) {
        pkv::set_error("unknown sequence %lld", (long long)seq_ids[i]);
        return PKV_ERR_UNKNOWN_SEQ;
      }
      if (seen[seq_ids[i]]++) return fail(PKV_ERR_INVALID_ARG, "a sequence appears twice in the batch");
    }
  }
  // batch order is priority order: the sequence preempted is always the
  // lowest-priority one still running (possibly the one being served)
  std::vector<char> alive(n_seqs, 1);
  int32_t last_alive = n_seqs - 1, n_cow = 0, n_pre = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    slots_out[i] = -1;
    if (!alive[i]) continue;
    for (;;) {
      auto it = pool->seqs.find(seq_ids[i]);
      bool cow = false;
      if (pkv::blocks_needed(pool, it->second, 1, &cow) <= pkv::available(pool)) {
        pkv::append_one(pool, seq_ids[i], it->second, 1, slots_out + i, cow_out, cow_cap, &n_cow,
                        nullptr);
        break;
      }
      while (!alive[last_alive]) --last_alive;
      const int32_t j = last_alive;
      pkv::free_seq_blocks(pool, pool->seqs.find(seq_ids[j]));
      alive[j] = 0;
      preempted_out[n_pre++] = seq_ids[j];
      if (j == i) break;
    }
  }
  if (n_cow_out) *n_cow_out = n_cow;
  if (n_preempted_out) *n_preempted_out = n_pre;
  return PKV_OK;
}

pkv_status pkv_seq_admit(pkv_pool* pool, int64_t seq_id, int32_t n_tokens, int32_t watermark_blocks,
                         int64_t* slots_out) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (n_tokens < 0 || watermark_blocks < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  if (n_tokens > 0 && !slots_out) return fail(PKV_ERR_INVALID_ARG, "slots_out is NULL");
  if (pool->seqs.count(seq_id)) {
    pkv::set_error("sequence %lld exists", (long long)seq_id);
    return PKV_ERR_INVALID_ARG;
  }
  const int64_t need = pkv::blocks_for(n_tokens, pool->block_size);
  if (need + watermark_blocks > pkv::available(pool)) {
    pkv::set_error("admitting %d tokens needs %lld blocks above a watermark of %d; %lld free",
                   n_tokens, (long long)need, watermark_blocks, (long long)pkv::available(pool));
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  pkv::Seq& s = pkv::add_seq(pool, seq_id, pkv::Seq{});
  int32_t n_cow = 0;
  return pkv::append_one(pool, seq_id, s, n_tokens, slots_out, nullptr, 0, &n_cow, nullptr);
}

}  // extern "C"

extern "C" const char* pkv_last_error(void) { return pkv::g_last_error.c_str(); }
