// Decode attention front end: argument checks, split-K partition choice,
// workspace layout, kernel selection and the split-K merge.
//
// Split-K (flash-decoding) is not described on the pages; it is how one
// sequence's positions are spread over several CTAs when the batch alone
// cannot fill the GPU.  Each split reports its running maximum m_i (log2
// domain), sum l_i and unnormalised output a_i; the merge forms
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  o = sum_i a_i 2^(m_i - M) / L,
// which equals the softmax over the union of the splits' positions.
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "attention.h"
#include "device_common.cuh"

namespace pkv {

// launch_decode_simt<KV, Q> is instantiated in attention_simt_<kv>_<q>.cu and
// launch_decode_tc<KV, Q> in attention_tc_<kv>_<q>.cu.
template <typename KV, typename Q>
pkv_status launch_decode_tc(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, cudaStream_t stream);

namespace {

constexpr int kMinPartition = 256;
constexpr int kMaxPartition = 8192;
constexpr int kMultiWavePartition = 4096;  // the smallest split when the pairs fill two waves
// Resident tensor-core split CTAs per SM: four for E4M3 caches (the
// head-columns kernel that every query group up to 8 takes), else three.
// Resident CTAs per SM of the tensor-core split kernel: four for E4M3, three
// otherwise; behind a shared-prefix pass 16-bit head_dim-128 caches take the
// narrow forms, eleven one-warp CTAs per SM at block size 16, six two-warp
// CTAs at 32.
int resident_split_ctas(const pkv_kv_desc* d, bool behind_prefix = false) {
  if (d->kv_dtype == PKV_E4M3) return 4;
  if (behind_prefix && d->head_dim == 128) return d->block_size == 16 ? 11 : 6;
  return 3;
}
constexpr int kDefaultSms = 152;       // used when no device can be queried

int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kDefaultSms;
  }
  if (dev < 64 && cache[dev].load() > 0) return cache[dev].load();
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return kDefaultSms;
  }
  if (dev < 64) cache[dev].store(sms);
  return sms;
}

// Automatic partition: the fewest tokens per split (a multiple of 64 and of
// the block size) for which the expected (sequence, head, split) units fit in
// one wave of resident CTAs, so that no unit waits for a slot.  Lengths are
// expected to spread evenly up to max_ctx, and each pair's last split to be
// half full.  With more (sequence, head) pairs than two waves of slots, the
// hardware balances the waves itself and splits cost merges; only the longest
// sequences are split in two (half of max_ctx, at least kMultiWavePartition),
// so that no single unit holds the tail of the last wave.
constexpr int32_t kTailPartition = 512;

int32_t auto_partition(int64_t num_seqs, int64_t num_kv_heads, int64_t max_ctx, int32_t block_size,
                       int ctas_per_sm) {
  const int64_t slots = static_cast<int64_t>(device_sms()) * ctas_per_sm;
  const int64_t pairs = num_seqs * num_kv_heads;
  const int64_t est_tokens = pairs * std::max<int64_t>(max_ctx, 1) / 2;
  const int32_t step = std::max<int32_t>(64, block_size);
  if (2 * slots <= pairs + 2) {
    const int64_t half = (std::max<int64_t>(max_ctx, 1) / 2 + step - 1) / step * step;
    return static_cast<int32_t>(std::min<int64_t>(kMaxPartition, std::max<int64_t>(kMultiWavePartition, half)));
  }
  const int64_t free_slots = slots - pairs / 2;
  int64_t p = (est_tokens + free_slots - 1) / free_slots;
  p = (p + step - 1) / step * step;
  return static_cast<int32_t>(std::min<int64_t>(kMaxPartition, std::max<int64_t>(kMinPartition, p)));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t counter_off, done_off, m_off, l_off, acc_off, bytes;
};

// Workspace: split-K arrival counters [B][N_kv] (zero between calls), then
// extra_ints more (behind a shared-prefix pass: the decode grid's exit
// count and the tail queue's claim counter), then the partial maxima, sums and unnormalised outputs, each part
// 256-byte aligned.  Nothing without splits.
WsLayout workspace_layout(int64_t num_seqs, int64_t num_q_heads, int64_t num_kv_heads,
                          int64_t splits, int64_t head_dim, int extra_ints = 0) {
  WsLayout w{};
  if (splits <= 1) return w;
  const size_t counters = static_cast<size_t>(num_seqs * num_kv_heads) + extra_ints;
  w.counter_off = 0;
  w.done_off = static_cast<size_t>(num_seqs * num_kv_heads) * sizeof(int);
  w.m_off = align_up(counters * sizeof(int), 256);
  const size_t n = static_cast<size_t>(num_seqs * num_q_heads * splits);
  w.l_off = w.m_off + align_up(n * sizeof(float), 256);
  w.acc_off = w.l_off + align_up(n * sizeof(float), 256);
  w.bytes = w.acc_off + align_up(n * head_dim * sizeof(float), 256);
  return w;
}


// Process-wide kernel choice (pkv_set_attention_kernel).
std::atomic<int> g_kernel_choice{PKV_KERNEL_AUTO};


// Whether the tensor-core kernel covers these sizes.
bool tc_supported(const pkv_kv_desc* d, int q_dtype, int group, int partition) {
  if (d->kv_dtype == PKV_F32) return false;
  if (group > 16) return false;
  if (partition / d->block_size > 1024) return false;
  if (static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * d->block_size > INT32_MAX) return false;
  if (d->kv_dtype == PKV_E4M3) return d->head_dim == 128 && (q_dtype == PKV_F16 || q_dtype == PKV_BF16);
  return d->head_dim == 128 || d->head_dim == 64;
}

// The split-K merge of the CUDA-core kernel, one CTA per (sequence, query
// head); a programmatic dependent of the decode kernel (it reads the
// partials after that grid has completed).
template <typename Q, int D>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int qh = blockIdx.x, seq = blockIdx.y;
  const int ctx = a.ctx_lens[seq];
  if (ctx < 0 || ctx > a.max_blocks * a.block_size) return;  // written by the decode kernel
  const int nsplit = max(1, (ctx + a.partition - 1) / a.partition);
  if (nsplit <= 1) return;
  const size_t base = (static_cast<size_t>(seq) * a.num_q_heads + qh) * a.max_splits;
  float M = -CUDART_INF_F;
  for (int i = 0; i < nsplit; ++i) M = fmaxf(M, a.ws_m[base + i]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float L = 0.f, A = 0.f;
    if (M != -CUDART_INF_F) {
      for (int i = 0; i < nsplit; ++i) {
        const float f = exp2f(a.ws_m[base + i] - M);
        L = fmaf(a.ws_l[base + i], f, L);
        A = fmaf(a.ws_acc[(base + i) * D + d], f, A);
      }
    } else {
      // no split attended a position: 0, or NaN from a split that failed
      for (int i = 0; i < nsplit; ++i) L += a.ws_l[base + i];
    }
    const float o = (L > 0.f || L != L) ? A / L : 0.f;
    store_elem<Q>(a.out, (static_cast<size_t>(seq) * a.num_q_heads + qh) * D + d, o);
  }
}

template <typename Q>
pkv_status launch_merge(const DecodeArgs& a, int head_dim, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.num_q_heads, a.num_seqs);
  cfg.blockDim = dim3(head_dim == 128 ? 128 : 64);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<Q, 128>, a)
                                        : cudaLaunchKernelEx(&cfg, merge_kernel<Q, 64>, a);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: merge launch", e);
  return check_launch("pkv_attention_decode (merge)");
}

// prefix_tokens: positions a shared-prefix pass covers (the decode kernel
// splits only the rest of each context).
pkv_status resolve_partition(int32_t requested, int32_t num_seqs, int32_t max_blocks,
                             const pkv_kv_desc* d, int32_t* out, int64_t prefix_tokens = 0) {
  if (requested < 0) return fail(PKV_ERR_INVALID_ARG, "partition_tokens is negative");
  if (requested > 0) {
    if (requested % 64 != 0 || requested % d->block_size != 0)
      return fail(PKV_ERR_INVALID_ARG, "partition_tokens must be a multiple of 64 and of block_size");
    *out = requested;
    return PKV_OK;
  }
  if (prefix_tokens > 0 && (d->kv_dtype == PKV_BF16 || d->kv_dtype == PKV_F16) && d->head_dim == 128 &&
      d->block_size == 16) {
    // past a shared prefix, 16-bit caches at block size 16 stream their
    // splits through the tail queue, whose units hold at most 32 tiles of 16
    // positions (a block id per lane); 512 positions per split measured
    // faster there than 256 (fewer partials and unit switches)
    *out = kTailPartition;
    return PKV_OK;
  }
  *out = auto_partition(num_seqs, d->num_kv_heads,
                        static_cast<int64_t>(max_blocks) * d->block_size - prefix_tokens,
                        d->block_size, resident_split_ctas(d, prefix_tokens > 0));
  return PKV_OK;
}

int64_t num_splits(int32_t max_blocks, int32_t block_size, int32_t partition,
                   int64_t prefix_tokens = 0) {
  const int64_t max_ctx = static_cast<int64_t>(max_blocks) * block_size - prefix_tokens;
  return std::max<int64_t>(1, (max_ctx + partition - 1) / partition);
}

// Shared-prefix pass geometry: the key ranges of the P prefix positions.
// A pass CTA holds a whole SM, and the decode kernel behind it streams the
// positions past the prefix on the SMs the pass leaves free, so the pass
// takes about a quarter of the SMs: each of the n_kv * ceil(rows / 256) row
// units gets that share of key ranges (at least one); ranges are whole
// 64-key tiles.
struct PrefixPlan {
  int32_t tokens = 0, key_splits = 0, split_tokens = 0, seqs_per_cta = 0;
};
PrefixPlan prefix_plan(int64_t num_seqs, int64_t group, int64_t num_kv_heads, int64_t prefix_tokens) {
  PrefixPlan p;
  if (prefix_tokens <= 0) return p;
  // a CTA's 256 query rows hold whole sequences (all G heads of each)
  p.seqs_per_cta = static_cast<int32_t>(256 / group);
  const int64_t units = (num_seqs + p.seqs_per_cta - 1) / p.seqs_per_cta * num_kv_heads;
  const int64_t tiles = (prefix_tokens + 63) / 64;
  const int64_t want =
      std::max<int64_t>(1, std::min<int64_t>(tiles, device_sms() / (4 * std::max<int64_t>(units, 1))));
  const int64_t per = (tiles + want - 1) / want;
  p.tokens = static_cast<int32_t>(prefix_tokens);
  p.split_tokens = static_cast<int32_t>(per * 64);
  p.key_splits = static_cast<int32_t>((tiles + per - 1) / per);
  return p;
}

// Whether the shared-prefix pass covers this call (else the prefix is read
// per sequence by the plain decode path).
bool prefix_pass_covers(const pkv_kv_desc* d, int q_dtype, float softmax_scale) {
  if (d->head_dim != 128 || !(softmax_scale > 0.f)) return false;
  if (d->kv_dtype == PKV_BF16) return q_dtype == PKV_BF16;
  if (d->kv_dtype == PKV_F16) return q_dtype == PKV_F16;
  return d->kv_dtype == PKV_E4M3 && (q_dtype == PKV_F16 || q_dtype == PKV_BF16);
}

// Everything a decode call decides before launching: the kernels, the
// partition, the split slots and the workspace layout.  sizing: for the
// workspace-size queries (q dtype and softmax scale taken as the ones that
// run the most kernels).
struct CallPlan {
  bool prefix_pass = false;
  PrefixPlan pp;
  int32_t partition = 0;
  int64_t splits = 1;   // tail splits + prefix key ranges
  WsLayout ws{};
};
pkv_status plan_call(const pkv_kv_desc* d, int q_dtype, float softmax_scale, int32_t num_seqs,
                     int32_t num_q_heads, int32_t max_blocks, int32_t partition_tokens,
                     int32_t prefix_blocks, CallPlan* out) {
  CallPlan c;
  const int group = num_q_heads / d->num_kv_heads;
  const int choice = g_kernel_choice.load();
  const bool rows_fit = static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * d->block_size <= INT32_MAX;
  c.prefix_pass = prefix_blocks > 0 && choice != PKV_KERNEL_SIMT && rows_fit &&
                  prefix_pass_covers(d, q_dtype, softmax_scale) && tc_supported(d, q_dtype, group, 64);
  if (c.prefix_pass)
    c.pp = prefix_plan(num_seqs, group, d->num_kv_heads, static_cast<int64_t>(prefix_blocks) * d->block_size);
  pkv_status st = resolve_partition(partition_tokens, num_seqs, max_blocks, d, &c.partition, c.pp.tokens);
  if (st != PKV_OK) return st;
  c.splits = num_splits(max_blocks, d->block_size, c.partition, c.pp.tokens) + c.pp.key_splits;
  c.ws = workspace_layout(num_seqs, num_q_heads, d->num_kv_heads, c.splits, d->head_dim,
                          c.prefix_pass ? 2 : 0);
  *out = c;
  return PKV_OK;
}

int sizing_q_dtype(const pkv_kv_desc* d) { return d->kv_dtype == PKV_E4M3 ? PKV_BF16 : d->kv_dtype; }

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool as a byte tensor of num_blocks * N_kv * T rows, read with the
// 128-byte swizzle: [rows][row_bytes] in boxes of T rows x 128 bytes (one
// slab), or, for 256-byte rows and whole_rows, [rows][2 slabs][128 bytes] in
// boxes of T whole rows.
pkv_status pool_map(CUtensorMap* map, const void* base, const pkv_kv_desc* d, bool whole_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(d->head_dim) * pkv_dtype_bytes(d->kv_dtype);
  const cuuint64_t rows = static_cast<cuuint64_t>(d->num_blocks) * d->num_kv_heads * d->block_size;
  const cuuint32_t t = static_cast<cuuint32_t>(d->block_size);
  CUresult r;
  if (row_bytes == 256 && whole_rows) {
    // (128 bytes, slab, row): one box carries both 128-byte slabs of T rows
    const cuuint64_t dims[3] = {128, 2, rows};
    const cuuint64_t strides[2] = {128, row_bytes};
    const cuuint32_t box[3] = {128, 2, t};
    const cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128, t};
    const cuuint32_t estr[2] = {1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
}  // namespace pkv

using namespace pkv;

extern "C" int32_t pkv_attention_partition(int32_t num_seqs, int32_t max_blocks,
                                           const pkv_kv_desc* desc, int32_t partition_tokens) {
  if (check_desc(desc) != PKV_OK || num_seqs < 0 || max_blocks < 0) return 0;
  int32_t p = 0;
  if (resolve_partition(partition_tokens, num_seqs, max_blocks, desc, &p) != PKV_OK) return 0;
  return p;
}

extern "C" size_t pkv_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                int32_t max_blocks, const pkv_kv_desc* desc,
                                                int32_t partition_tokens) {
  if (check_desc(desc) != PKV_OK || num_seqs <= 0 || num_q_heads <= 0 || max_blocks <= 0) return 0;
  if (num_q_heads % desc->num_kv_heads != 0) return 0;
  CallPlan c;
  if (plan_call(desc, sizing_q_dtype(desc), 1.f, num_seqs, num_q_heads, max_blocks, partition_tokens,
                0, &c) != PKV_OK)
    return 0;
  return c.ws.bytes;
}

namespace pkv {
size_t attention_counter_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks,
                               const pkv_kv_desc* desc, int32_t partition_tokens) {
  if (check_desc(desc) != PKV_OK || num_seqs <= 0 || num_q_heads <= 0 || max_blocks <= 0) return 0;
  if (num_q_heads % desc->num_kv_heads != 0) return 0;
  CallPlan c;
  if (plan_call(desc, sizing_q_dtype(desc), 1.f, num_seqs, num_q_heads, max_blocks, partition_tokens,
                0, &c) != PKV_OK)
    return 0;
  return c.ws.bytes ? c.ws.m_off : 0;
}
}  // namespace pkv

extern "C" pkv_status pkv_set_attention_kernel(int32_t kind) {
  if (kind != PKV_KERNEL_AUTO && kind != PKV_KERNEL_SIMT && kind != PKV_KERNEL_TENSOR_CORE)
    return fail(PKV_ERR_INVALID_ARG, "unknown attention kernel kind");
  g_kernel_choice.store(kind);
  return PKV_OK;
}

namespace pkv {
namespace {
// Decode attention, optionally preceded by the step's slot write (k_new set):
// fused into the tensor-core split kernel, else a small write kernel first.
pkv_status decode_impl(void* out, const void* q, int32_t q_dtype, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables, int32_t max_blocks,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       const pkv_kv_desc* desc, float softmax_scale, float k_scale, float v_scale,
                       int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                       void* stream, const void* k_new, const void* v_new, float k_inv,
                       float v_inv, int32_t prefix_blocks = 0) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_q_heads <= 0 || max_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size or no query heads");
  if (prefix_blocks < 0 || prefix_blocks > max_blocks)
    return fail(PKV_ERR_INVALID_ARG, "prefix_blocks outside [0, max_blocks]");
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return fail(PKV_ERR_UNSUPPORTED, "more than 65535 sequences per call");
  if (max_blocks == 0) return fail(PKV_ERR_INVALID_ARG, "max_blocks is 0");
  if (num_q_heads % desc->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  for (const void* p : {static_cast<const void*>(out), q, k_cache, v_cache})
    if (!aligned(p, 16)) return fail(PKV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PKV_ERR_INVALID_ARG, "tables misaligned");
  if (static_cast<int64_t>(max_blocks) * desc->block_size > (int64_t{1} << 30))
    return fail(PKV_ERR_UNSUPPORTED, "context longer than 2^30 tokens");
  if (!(softmax_scale == softmax_scale)) return fail(PKV_ERR_INVALID_ARG, "softmax_scale is NaN");

  const int kv = desc->kv_dtype;
  const bool pair_ok = (kv == PKV_F32 && q_dtype == PKV_F32) ||
                       (kv == PKV_F16 && q_dtype == PKV_F16) ||
                       (kv == PKV_BF16 && q_dtype == PKV_BF16) ||
                       (kv == PKV_E4M3 && (q_dtype == PKV_F16 || q_dtype == PKV_BF16));
  if (!pair_ok) return fail(PKV_ERR_INVALID_ARG, "unsupported (kv_dtype, q_dtype) pair");

  const int group = num_q_heads / desc->num_kv_heads;
  int gm = 1;
  while (gm < group) gm = gm == 1 ? 4 : gm * 2;
  if (gm > 16) return fail(PKV_ERR_UNSUPPORTED, "more than 16 query heads per KV head");
  const int choice = g_kernel_choice.load();

  // A declared shared prefix runs the prefix pass where it covers the shape
  // under the tensor-core decode kernels; otherwise the prefix is read per
  // sequence like the rest of the context (same attention).
  CallPlan plan;
  st = plan_call(desc, q_dtype, softmax_scale, num_seqs, num_q_heads, max_blocks, partition_tokens,
                 prefix_blocks, &plan);
  if (st != PKV_OK) return st;
  const bool prefix_pass = plan.prefix_pass;
  const PrefixPlan pp = plan.pp;
  const int32_t partition = plan.partition;
  const int64_t splits = plan.splits;
  if (splits > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many splits");
  const WsLayout ws = plan.ws;
  if (ws.bytes > 0) {
    if (!workspace || workspace_bytes < ws.bytes)
      return fail(PKV_ERR_INVALID_ARG, "workspace missing or smaller than the workspace size call");
    if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  int* status = device_status_word(&st);
  if (!status) return st;

  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.tables = block_tables;
  a.ctx_lens = context_lens;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  const bool partials = ws.bytes > ws.m_off;
  a.ws_m = partials ? reinterpret_cast<float*>(wsb + ws.m_off) : nullptr;
  a.ws_l = partials ? reinterpret_cast<float*>(wsb + ws.l_off) : nullptr;
  a.ws_acc = partials ? reinterpret_cast<float*>(wsb + ws.acc_off) : nullptr;
  a.counters = ws.bytes ? reinterpret_cast<int*>(wsb + ws.counter_off) : nullptr;
  a.max_blocks = max_blocks;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = desc->num_kv_heads;
  a.group = group;
  a.num_blocks = desc->num_blocks;
  a.block_size = desc->block_size;
  a.partition = partition;
  a.max_splits = static_cast<int32_t>(splits);
  const bool fp8 = kv == PKV_E4M3;
  a.qk_scale = softmax_scale * (fp8 ? k_scale : 1.0f) * 1.4426950408889634f;
  a.v_scale = fp8 ? v_scale : 1.0f;
  a.head_scales = desc->head_scales;
  a.softmax_scale = softmax_scale;
  a.prefix_tokens = pp.tokens;
  a.prefix_splits = pp.key_splits;
  a.done = prefix_pass ? reinterpret_cast<int*>(wsb + ws.done_off) : nullptr;
  a.tail_queue = choice == PKV_KERNEL_AUTO ? 1 : 0;
  a.status = status;
  a.wait_ns = stage_wait_limit_ns();

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = desc->head_dim;
  const bool tc_ok = tc_supported(desc, q_dtype, group, partition);
  if (choice == PKV_KERNEL_TENSOR_CORE && !tc_ok)
    return fail(PKV_ERR_UNSUPPORTED, "the tensor-core kernel does not cover these sizes");
  if (prefix_pass && !tc_ok)
    return fail(PKV_ERR_UNSUPPORTED, "partition too long for the tensor-core kernel");
  if (k_new) {
    if (tc_ok && choice != PKV_KERNEL_SIMT) {
      a.k_new = k_new;  // fused into the split kernel
      a.v_new = v_new;
      a.k_inv = kv == PKV_E4M3 ? k_inv : 1.0f;
      a.v_inv = kv == PKV_E4M3 ? v_inv : 1.0f;
    } else {
      st = launch_write_last(const_cast<void*>(k_cache), const_cast<void*>(v_cache), k_new, v_new,
                             q_dtype, k_inv, v_inv, block_tables, max_blocks, context_lens,
                             num_seqs, desc, s);
      if (st != PKV_OK) return st;
    }
  }
  if (prefix_pass) {
    // the prefix pass first: its CTAs let the decode kernel start once they
    // have all begun, on the SMs the pass leaves free; both write partials,
    // which the merge kernel after the decode kernel combines
    PrefillArgs pa{};
    pa.q = q;
    pa.tables = block_tables;
    pa.max_blocks = max_blocks;
    pa.num_seqs = num_seqs;
    pa.total_q = num_seqs * group;
    pa.num_q_heads = num_q_heads;
    pa.num_kv_heads = desc->num_kv_heads;
    pa.group = group;
    pa.num_blocks = desc->num_blocks;
    pa.qk_scale = a.qk_scale;
    pa.v_scale = a.v_scale;
    pa.head_scales = desc->head_scales;
    pa.softmax_scale = softmax_scale;
    pa.status = status;
    pa.sp_rows = num_seqs * group;
    pa.sp_tokens = pp.tokens;
    pa.sp_split = pp.split_tokens;
    pa.sp_slot0 = static_cast<int32_t>(splits) - pp.key_splits;
    pa.max_splits = static_cast<int32_t>(splits);
    pa.ws_m = a.ws_m;
    pa.ws_l = a.ws_l;
    pa.ws_acc = a.ws_acc;
    pa.sp_seqs = pp.seqs_per_cta;
    CUtensorMap pkmap, pvmap;
    st = pool_map(&pkmap, k_cache, desc, false);
    if (st == PKV_OK) st = pool_map(&pvmap, v_cache, desc, false);
    if (st != PKV_OK) return st;
    const int T = desc->block_size;
    switch (kv) {
      case PKV_F16: st = launch_shared_prefix_pass<F16, F16>(pa, T, pp.key_splits, pkmap, pvmap, s); break;
      case PKV_BF16: st = launch_shared_prefix_pass<BF16, BF16>(pa, T, pp.key_splits, pkmap, pvmap, s); break;
      default:
        st = q_dtype == PKV_F16 ? launch_shared_prefix_pass<E4M3, F16>(pa, T, pp.key_splits, pkmap, pvmap, s)
                                : launch_shared_prefix_pass<E4M3, BF16>(pa, T, pp.key_splits, pkmap, pvmap, s);
    }
    if (st != PKV_OK) return st;
  }
  if (tc_ok && choice != PKV_KERNEL_SIMT) {
    CUtensorMap kmap, vmap;
    st = pool_map(&kmap, k_cache, desc);
    if (st == PKV_OK) st = pool_map(&vmap, v_cache, desc);
    if (st != PKV_OK) return st;
    switch (kv) {
      case PKV_F16: st = launch_decode_tc<F16, F16>(a, D, kmap, vmap, s); break;
      case PKV_BF16: st = launch_decode_tc<BF16, BF16>(a, D, kmap, vmap, s); break;
      default:
        st = q_dtype == PKV_F16 ? launch_decode_tc<E4M3, F16>(a, D, kmap, vmap, s)
                                : launch_decode_tc<E4M3, BF16>(a, D, kmap, vmap, s);
    }
    // behind a shared-prefix pass every partial is merged by the merge kernel
    if (st != PKV_OK || !prefix_pass) return st;
    return q_dtype == PKV_F16 ? launch_prefix_merge<F16>(a, s) : launch_prefix_merge<BF16>(a, s);
  }
  switch (kv) {
    case PKV_F32: st = launch_decode_simt<F32, F32>(a, D, gm, s); break;
    case PKV_F16: st = launch_decode_simt<F16, F16>(a, D, gm, s); break;
    case PKV_BF16: st = launch_decode_simt<BF16, BF16>(a, D, gm, s); break;
    case PKV_E4M3:
      st = q_dtype == PKV_F16 ? launch_decode_simt<E4M3, F16>(a, D, gm, s)
                              : launch_decode_simt<E4M3, BF16>(a, D, gm, s);
      break;
  }
  if (st != PKV_OK || splits <= 1) return st;
  switch (q_dtype) {
    case PKV_F32: return launch_merge<F32>(a, D, s);
    case PKV_F16: return launch_merge<F16>(a, D, s);
    default: return launch_merge<BF16>(a, D, s);
  }
}
}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_attention_decode(void* out, const void* q, int32_t q_dtype,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, int32_t max_blocks,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, const pkv_kv_desc* desc,
                                           float softmax_scale, float k_scale, float v_scale,
                                           int32_t partition_tokens, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, q_dtype, k_cache, v_cache, block_tables, max_blocks, context_lens,
                     num_seqs, num_q_heads, desc, softmax_scale, k_scale, v_scale, partition_tokens,
                     workspace, workspace_bytes, stream, nullptr, nullptr, 1.0f, 1.0f);
}

extern "C" pkv_status pkv_decode_step(void* out, const void* q, int32_t q_dtype, void* k_cache,
                                      void* v_cache, const void* k_new, const void* v_new,
                                      const int32_t* block_tables, int32_t max_blocks,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, const pkv_kv_desc* desc,
                                      float softmax_scale, float k_scale, float v_scale,
                                      float k_inv_scale, float v_inv_scale,
                                      int32_t partition_tokens, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "k_new or v_new is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  return decode_impl(out, q, q_dtype, k_cache, v_cache, block_tables, max_blocks, context_lens,
                     num_seqs, num_q_heads, desc, softmax_scale, k_scale, v_scale, partition_tokens,
                     workspace, workspace_bytes, stream, k_new, v_new, k_inv_scale, v_inv_scale);
}

extern "C" size_t pkv_shared_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                    int32_t max_blocks, const pkv_kv_desc* desc,
                                                    int32_t prefix_blocks, int32_t partition_tokens) {
  if (check_desc(desc) != PKV_OK || num_seqs <= 0 || num_q_heads <= 0 || max_blocks <= 0) return 0;
  if (prefix_blocks < 0 || prefix_blocks > max_blocks || num_q_heads % desc->num_kv_heads != 0) return 0;
  // the size the prefix pass needs; calls that run without it need no more
  // than the plain call
  CallPlan c;
  if (plan_call(desc, sizing_q_dtype(desc), 1.f, num_seqs, num_q_heads, max_blocks, partition_tokens,
                prefix_blocks, &c) != PKV_OK)
    return 0;
  return std::max(c.ws.bytes, pkv_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc,
                                                            partition_tokens));
}

extern "C" pkv_status pkv_attention_decode_shared_prefix(
    void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc, int32_t prefix_blocks,
    float softmax_scale, float k_scale, float v_scale, int32_t partition_tokens, void* workspace,
    size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, q_dtype, k_cache, v_cache, block_tables, max_blocks, context_lens,
                     num_seqs, num_q_heads, desc, softmax_scale, k_scale, v_scale, partition_tokens,
                     workspace, workspace_bytes, stream, nullptr, nullptr, 1.0f, 1.0f, prefix_blocks);
}

extern "C" pkv_status pkv_decode_step_shared_prefix(
    void* out, const void* q, int32_t q_dtype, void* k_cache, void* v_cache, const void* k_new,
    const void* v_new, const int32_t* block_tables, int32_t max_blocks,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc,
    int32_t prefix_blocks, float softmax_scale, float k_scale, float v_scale, float k_inv_scale,
    float v_inv_scale, int32_t partition_tokens, void* workspace, size_t workspace_bytes,
    void* stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return fail(PKV_ERR_INVALID_ARG, "k_new or v_new is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  return decode_impl(out, q, q_dtype, k_cache, v_cache, block_tables, max_blocks, context_lens,
                     num_seqs, num_q_heads, desc, softmax_scale, k_scale, v_scale, partition_tokens,
                     workspace, workspace_bytes, stream, k_new, v_new, k_inv_scale, v_inv_scale,
                     prefix_blocks);
}
