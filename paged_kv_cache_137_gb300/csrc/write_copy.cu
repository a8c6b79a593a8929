// Slot write and copy-on-write block copy.
//
// Slot write: each decode step writes the new tokens' keys and values into the
// slots the allocator reserved (foundry page on paged block allocation, "In
// and out": the number of new tokens about to be written).  Block copy: a
// shared block is copied before a branch writes into it (same page,
// "Concept"; katajob Q&A, "Sharing, the second dividend").
//
// Both are tiny, latency-bound kernels: 16-byte vector accesses, one thread
// per 8-element unit of a (token, head) row for the write and one CTA per
// (pair, layer, K|V) tile for the copy.  The copy takes its pairs and layer
// pointers as kernel parameters, so it needs no device-side staging buffer.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "device_common.cuh"

namespace pkv {
namespace {

// The E4M3 inverse scale of K (which = 0) or V of KV head h: the per-head
// table's rows 2 and 3 when there is one, else the per-tensor value.
__device__ __forceinline__ float inv_of(const float* head_scales, const float* inv_scale, int n_kv,
                                        int which, int h) {
  return head_scales ? head_scales[(2 + which) * n_kv + h] : inv_scale[which];
}

struct WriteArgs {
  void* cache[2];       // K, V caches
  const void* src[2];   // K, V inputs [n_tokens][n_kv][D]
  float inv_scale[2];
  const float* head_scales;  // E4M3 per-head scales [4][n_kv], or NULL
  const int64_t* slots;
  int64_t n_tokens;
  int32_t n_kv, head_dim, block_size, num_blocks;
};

// One unit = 8 consecutive elements of one (token, head) row.
template <typename Src, typename Dst>
__global__ void __launch_bounds__(256) write_kernel(const WriteArgs a) {
  // a decode kernel launched after this one as a programmatic dependent may
  // be scheduled now; it waits for this grid's completion before its reads
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int which = blockIdx.y;  // 0 = K, 1 = V
  const int units_per_row = a.head_dim / 8;
  const int64_t units = a.n_tokens * a.n_kv * units_per_row;
  const int64_t limit = static_cast<int64_t>(a.num_blocks) * a.block_size;
  for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < units;
       u += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tok = u / (a.n_kv * units_per_row);
    const int rem = static_cast<int>(u - tok * a.n_kv * units_per_row);
    const int h = rem / units_per_row;
    const int d0 = (rem - h * units_per_row) * 8;
    const int64_t slot = a.slots[tok];
    if (slot < 0 || slot >= limit) continue;
    const int64_t blk = slot / a.block_size;
    const int off = static_cast<int>(slot - blk * a.block_size);
    const size_t src_idx = (static_cast<size_t>(tok) * a.n_kv + h) * a.head_dim + d0;
    const size_t dst_idx =
        ((static_cast<size_t>(blk) * a.n_kv + h) * a.block_size + off) * a.head_dim + d0;
    store8<Src, Dst>(static_cast<const typename Src::raw*>(a.src[which]) + src_idx,
                     static_cast<typename Dst::raw*>(a.cache[which]) + dst_idx,
                     inv_of(a.head_scales, a.inv_scale, a.n_kv, which, h));
  }
}

// The step's token of each sequence: K/V row [n_kv][D] of batch row s written
// at logical position ctx_s - 1 through its block table (nothing for a
// length outside [1, max_blocks * T] or a table entry outside the pool).
struct WriteLastArgs {
  void* cache[2];
  const void* src[2];   // [B][n_kv][D]
  float inv_scale[2];
  const float* head_scales;
  const int32_t* tables;
  const int32_t* ctx_lens;
  int32_t max_blocks, n_kv, head_dim, block_size, num_blocks;
};

template <typename Src, typename Dst>
__global__ void __launch_bounds__(128) write_last_kernel(const WriteLastArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s = blockIdx.x, which = blockIdx.y;
  const int ctx = a.ctx_lens[s];
  if (ctx < 1 || ctx > a.max_blocks * a.block_size) return;
  const int p = ctx - 1;
  const int blk = a.tables[static_cast<size_t>(s) * a.max_blocks + p / a.block_size];
  if (blk < 0 || blk >= a.num_blocks) return;
  const int units = a.n_kv * (a.head_dim / 8);
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int h = u / (a.head_dim / 8), d0 = (u % (a.head_dim / 8)) * 8;
    const size_t src_idx = (static_cast<size_t>(s) * a.n_kv + h) * a.head_dim + d0;
    const size_t dst_idx =
        ((static_cast<size_t>(blk) * a.n_kv + h) * a.block_size + p % a.block_size) * a.head_dim + d0;
    store8<Src, Dst>(static_cast<const typename Src::raw*>(a.src[which]) + src_idx,
                     static_cast<typename Dst::raw*>(a.cache[which]) + dst_idx,
                     inv_of(a.head_scales, a.inv_scale, a.n_kv, which, h));
  }
}

constexpr int kMaxCopyLayers = 128;
constexpr int kMaxCopyPairs = 1024;

struct CopyArgs {
  void* k[kMaxCopyLayers];
  void* v[kMaxCopyLayers];
  int32_t src[kMaxCopyPairs];
  int32_t dst[kMaxCopyPairs];
  int64_t block_bytes;  // bytes of one block in one layer's K (or V) tensor
};

// grid: (pair, layer, K|V); each CTA copies one block of one tensor.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const __grid_constant__ CopyArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int pair = blockIdx.x, layer = blockIdx.y;
  uint8_t* base = static_cast<uint8_t*>(blockIdx.z == 0 ? a.k[layer] : a.v[layer]);
  const uint4* s = reinterpret_cast<const uint4*>(base + a.src[pair] * a.block_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + a.dst[pair] * a.block_bytes);
  const int64_t n = a.block_bytes / 16;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

template <typename Src, typename Dst>
pkv_status launch_write(const WriteArgs& a, cudaStream_t st) {
  const int64_t units = a.n_tokens * a.n_kv * (a.head_dim / 8);
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((units + threads - 1) / threads, 4096);
  static std::atomic<uint64_t> carveout{0};
  prefer_max_shared(write_kernel<Src, Dst>, carveout);
  write_kernel<Src, Dst><<<dim3(static_cast<unsigned>(blocks), 2), threads, 0, st>>>(a);
  return check_launch("pkv_write");
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_write(void* k_cache, void* v_cache, const void* k, const void* v,
                                int32_t src_dtype, const int64_t* slot_mapping, int32_t n_tokens,
                                const pkv_kv_desc* desc, float k_inv_scale, float v_inv_scale,
                                void* stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (n_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "n_tokens is negative");
  if (n_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !k || !v || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  for (const void* p : {static_cast<const void*>(k_cache), static_cast<const void*>(v_cache), k, v})
    if (!aligned(p, 16)) return fail(PKV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping misaligned");
  WriteArgs a{};
  a.cache[0] = k_cache;
  a.cache[1] = v_cache;
  a.src[0] = k;
  a.src[1] = v;
  a.inv_scale[0] = k_inv_scale;
  a.inv_scale[1] = v_inv_scale;
  a.head_scales = desc->head_scales;
  a.slots = slot_mapping;
  a.n_tokens = n_tokens;
  a.n_kv = desc->num_kv_heads;
  a.head_dim = desc->head_dim;
  a.block_size = desc->block_size;
  a.num_blocks = desc->num_blocks;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int kv = desc->kv_dtype;
  if (kv == PKV_E4M3) {
    switch (src_dtype) {
      case PKV_F32: return launch_write<F32, E4M3>(a, s);
      case PKV_F16: return launch_write<F16, E4M3>(a, s);
      case PKV_BF16: return launch_write<BF16, E4M3>(a, s);
      default: return fail(PKV_ERR_INVALID_ARG, "src_dtype must be F32, F16 or BF16");
    }
  }
  if (src_dtype != kv)
    return fail(PKV_ERR_INVALID_ARG, "a 16/32-bit cache needs src_dtype == kv_dtype");
  switch (kv) {
    case PKV_F32: return launch_write<F32, F32>(a, s);
    case PKV_F16: return launch_write<F16, F16>(a, s);
    case PKV_BF16: return launch_write<BF16, BF16>(a, s);
  }
  return fail(PKV_ERR_INVALID_ARG, "unknown kv_dtype");
}

extern "C" pkv_status pkv_copy_blocks(void* const* k_caches, void* const* v_caches,
                                      int32_t num_layers, const int32_t* src_dst, int32_t n_pairs,
                                      const pkv_kv_desc* desc, void* stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (n_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "n_pairs is negative");
  if (n_pairs == 0) return PKV_OK;
  if (num_layers <= 0 || num_layers > kMaxCopyLayers)
    return fail(PKV_ERR_INVALID_ARG, "num_layers must be in [1, 128]");
  if (!k_caches || !v_caches || !src_dst) return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  for (int32_t l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l]) return fail(PKV_ERR_INVALID_ARG, "NULL layer pointer");
    if (!aligned(k_caches[l], 16) || !aligned(v_caches[l], 16))
      return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  }
  for (int32_t i = 0; i < 2 * n_pairs; ++i)
    if (src_dst[i] < 0 || src_dst[i] >= desc->num_blocks)
      return fail(PKV_ERR_INVALID_ARG, "block id out of range");
  CopyArgs a;
  for (int32_t l = 0; l < num_layers; ++l) {
    a.k[l] = k_caches[l];
    a.v[l] = v_caches[l];
  }
  a.block_bytes = static_cast<int64_t>(desc->num_kv_heads) * desc->block_size * desc->head_dim *
                  pkv_dtype_bytes(desc->kv_dtype);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static std::atomic<uint64_t> carveout{0};
  prefer_max_shared(copy_blocks_kernel, carveout);
  for (int32_t base = 0; base < n_pairs; base += kMaxCopyPairs) {
    const int32_t n = std::min(kMaxCopyPairs, n_pairs - base);
    for (int32_t i = 0; i < n; ++i) {
      a.src[i] = src_dst[2 * (base + i)];
      a.dst[i] = src_dst[2 * (base + i) + 1];
    }
    copy_blocks_kernel<<<dim3(n, num_layers, 2), 256, 0, s>>>(a);
    st = check_launch("pkv_copy_blocks");
    if (st != PKV_OK) return st;
  }
  return PKV_OK;
}

namespace pkv {

template <typename Src, typename Dst>
static pkv_status launch_write_last_dt(const WriteLastArgs& a, int32_t num_seqs, cudaStream_t st) {
  static std::atomic<uint64_t> carveout{0};
  prefer_max_shared(write_last_kernel<Src, Dst>, carveout);
  write_last_kernel<Src, Dst><<<dim3(num_seqs, 2), 128, 0, st>>>(a);
  return check_launch("pkv_decode_step (write)");
}

pkv_status launch_write_last(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             int32_t src_dtype, float k_inv_scale, float v_inv_scale,
                             const int32_t* tables, int32_t max_blocks, const int32_t* ctx_lens,
                             int32_t num_seqs, const pkv_kv_desc* desc, cudaStream_t st) {
  WriteLastArgs a{};
  a.cache[0] = k_cache;
  a.cache[1] = v_cache;
  a.src[0] = k_new;
  a.src[1] = v_new;
  a.inv_scale[0] = k_inv_scale;
  a.inv_scale[1] = v_inv_scale;
  a.head_scales = desc->head_scales;
  a.tables = tables;
  a.ctx_lens = ctx_lens;
  a.max_blocks = max_blocks;
  a.n_kv = desc->num_kv_heads;
  a.head_dim = desc->head_dim;
  a.block_size = desc->block_size;
  a.num_blocks = desc->num_blocks;
  const int kv = desc->kv_dtype;
  if (kv == PKV_E4M3) {
    switch (src_dtype) {
      case PKV_F32: return launch_write_last_dt<F32, E4M3>(a, num_seqs, st);
      case PKV_F16: return launch_write_last_dt<F16, E4M3>(a, num_seqs, st);
      case PKV_BF16: return launch_write_last_dt<BF16, E4M3>(a, num_seqs, st);
      default: return fail(PKV_ERR_INVALID_ARG, "k_new dtype must be F32, F16 or BF16");
    }
  }
  if (src_dtype != kv) return fail(PKV_ERR_INVALID_ARG, "a 16/32-bit cache needs k_new of its dtype");
  switch (kv) {
    case PKV_F32: return launch_write_last_dt<F32, F32>(a, num_seqs, st);
    case PKV_F16: return launch_write_last_dt<F16, F16>(a, num_seqs, st);
    case PKV_BF16: return launch_write_last_dt<BF16, BF16>(a, num_seqs, st);
  }
  return fail(PKV_ERR_INVALID_ARG, "unknown kv_dtype");
}

}  // namespace pkv
