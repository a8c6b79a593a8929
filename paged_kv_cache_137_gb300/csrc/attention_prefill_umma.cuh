// Prefill attention on the 5th-generation tensor cores (tcgen05 / UMMA with
// TMEM accumulators), 16-bit caches, head_dim 128.
//
// Same computation as prefill_tc_kernel (the chunk's queries attend causally
// over the cached positions through the block table); this is the GB300 form:
//  * One CTA per (pair of 128-query tiles, query head, sequence), 10 warps:
//      warps 0-3  softmax of query tile A: thread r owns row r (TMEM lane r);
//      warps 4-7  softmax of query tile B (the next 128 positions);
//      warp 8     TMA producer of the K/V ring, TMEM allocation;
//      warp 9     MMA issuer (one thread).
//    Both query tiles use every K/V tile the ring brings (B's last one or
//    two only it), and each SM sub-partition holds two softmax warps, one
//    per tile, so one works while the other waits on its loads.
//  * Per 64-key tile t:  S_t = Q K_t^T (M 128, N 64, K 128: 8 UMMAs) into one of
//    two TMEM S buffers; the softmax threads read their S row (tcgen05.ld),
//    apply the causal mask and the online softmax, and write P_t (16-bit
//    pairs) back over the S buffer they read (tcgen05.st); then
//    O += P_t V_t (M 128, N 128, K 64: 4 UMMAs with A read from TMEM, V read
//    N-major from shared memory) into TMEM.  P never touches shared memory.
//    S_{t+2} is issued once P_t V_t is done (P_t occupies S_{t+2}'s buffer),
//    so the tensor core works two tiles ahead while the softmax threads work
//    on this one, and a K/V load that is late holds up only the S product
//    that needs it.
//  * With up to 256 (sequence, query-tile pair) units the grid is (query
//    head, unit rank): each CTA ranks the units by the key tiles they read
//    and takes the one of its rank, so long units are dispatched first.
//  * O stays in TMEM.  A row's reference maximum moves only when the running
//    maximum exceeds it by more than 8 (log2 units): then that row of O is
//    read, scaled and written back (after the previous P V has completed).
//    P = 2^(s - m_ref) <= 2^8 in between; the final O / l uses the same
//    reference, so the result is the softmax whichever references were used.
//  * Q is loaded by the softmax threads into the 128-byte-swizzled K-major
//    layout; K and V arrive by 2-D TMA boxes of T rows x 128 bytes per
//    (block, slab) into a 5-stage ring, the layout the UMMA shared-memory
//    descriptors describe.
//  * The softmax takes the row maximum on the raw scores and computes each
//    exponent as 2^(s * scale - m) with one FFMA, which needs scale > 0 (the
//    host sends other scales to the mma.sync kernel).
//  * V rows at positions >= ctx are zeroed in shared memory before P V
//    (0 * NaN would poison the product; the mask already zeroes P there).
//  * Every mbarrier wait is bounded; a CTA whose wait gives up writes NaN
//    rows, waits (bounded) for its copies and MMAs in flight, and frees its
//    TMEM before it exits.
//
// Shared-prefix pass (kCasc): the same pipeline computes, for one KV head,
// the attention of every (sequence, query head) row of a decode batch (row
// r = s * G + j, M = num_seqs * G rows, two 128-row tiles per CTA) over one
// key range of the positions [0, P) that all sequences share, read through
// table row 0 (the katajob Q&A, "Sharing, the second dividend": sequences
// that share a prompt list the same physical blocks; "PagedAttention Memory
// Management", "Complex Topologies and Memory Sharing").  Nothing is masked
// but the end of the range, and each row leaves its partial result (running
// maximum, sum, unnormalised output times the V scale) in a split slot of the
// decode workspace; the merge kernel after the decode kernel combines it with
// the rest of the sequence's context.  The CTAs let the decode kernel launch
// as soon as they have all started (griddepcontrol.launch_dependents after
// their own wait), on the SMs this grid leaves free.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "attention.h"
#include "attention_tc.cuh"
#include "device_common.cuh"

namespace pkv {
namespace tc {
namespace umma {

constexpr int kRows = 128;       // query rows per query tile (UMMA M)
constexpr int kKeys = 64;        // keys per tile (UMMA N of S)
constexpr int kStages = 5;       // K/V ring depth: loads run up to 4 tiles ahead
constexpr int kThreadsU = 320;   // 2 x 4 softmax warps, the producer warp, the MMA warp
constexpr int kTmemCols = 512;   // per query tile X: S0 [256X, +64), S1 [+64, +64), O [+128, +128);
                                 // P_t (16-bit pairs) overwrites the first 32 columns of its S buffer
constexpr int kQBytes = kRows * 256;          // two slabs of 128 rows x 128 bytes
constexpr int kSlab = kKeys * 128;            // one slab of a K or V tile
constexpr int kKVBytes = 2 * kSlab;           // K (or V) tile: 64 rows x 256 bytes
constexpr int kStageBytes = 2 * kKVBytes;     // K then V
constexpr float kRescaleLog2 = 8.f;

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// D[tmem] (+)= A[smem desc] x B[smem desc], kind::f16, one CTA.
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem desc]: A (M rows = TMEM lanes, two 16-bit K
// elements per 32-bit column) read from tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once every UMMA this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, -inf gives 0), for the softmax exponentials.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting
// for them (tmem_wait_ld before use).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1, layout
// type 2 (128-byte swizzle).  K-major operands: rows of 128 bytes, 8-row
// groups SBO apart (the leading offset is not used).  N-major operands
// (V): LBO between 64-element column blocks, SBO between 8-row groups.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t{1} << 46;
  d |= uint64_t{2} << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (or both f16), A K-major, B K-major or N-major, shape M x N.
constexpr uint32_t idesc(bool bf, int M, int N, bool b_n_major) {
  return (1u << 4) | (static_cast<uint32_t>(bf) << 7) | (static_cast<uint32_t>(bf) << 10) |
         (static_cast<uint32_t>(b_n_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// block of 128-byte rows (1024-byte aligned).
__device__ __forceinline__ uint32_t sw(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

constexpr int kMaxRanked = 256;   // units ranked in the kernel (longest first)

// The (sequence, query-tile pair) unit of rank `rank` when the units are
// ordered by work (the key tiles both query tiles read), longest first, ties
// in sequence order.  The hardware dispatches CTAs in grid order, so the
// long units start first and the short ones fill the gaps at the end (the
// longest-processing-time rule).  Every CTA computes the same order from the
// lengths: sequence t is thread t's, at most kMaxRanked units in all.
// Returns the sequence (or -1: no unit of that rank) and the pair index.
template <int T>
__device__ __forceinline__ int ranked_unit(const PrefillArgs& a, int rank, int* scratch, int* pair_out) {
  int* s_work = scratch;                     // [kMaxRanked]
  int* s_seq = s_work + kMaxRanked;          // [kMaxRanked]
  int* s_pair = s_seq + kMaxRanked;          // [kMaxRanked]
  int* s_wsum = s_pair + kMaxRanked;         // [8] unit counts of the warps' sequences
  int* s_pick = s_wsum + 8;                  // [2]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int np = 0, first = 0, n = 0;
  bool bad = false;
  if (tid < a.num_seqs) {
    const int ctx = a.ctx_lens[tid];
    const int q0 = a.query_start[tid];
    n = a.query_start[tid + 1] - q0;
    if (!(q0 < 0 || n <= 0 || q0 + n > a.total_q)) {
      const int ntq = (n + kRows - 1) / kRows;
      bad = ctx < 0 || ctx > a.max_blocks * T || n > ctx || (ntq + 1) / 2 > a.max_q_tiles;
      np = bad ? 1 : (ntq + 1) / 2;  // an invalid sequence: one unit that writes its NaN rows
      first = ctx - n;
    }
  }
  // offset of sequence tid's units: a scan within each of the first 8 warps
  // (num_seqs <= kMaxRanked = 256), then over the warps' totals
  int incl = np;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (warp < 8 && lane == 31) s_wsum[warp] = incl;
  if (tid < 2) s_pick[tid] = -1;
  __syncthreads();
  int base = 0, units = 0;
  for (int w = 0; w < 8; ++w) {
    base += w < warp ? s_wsum[w] : 0;
    units += s_wsum[w];
  }
  if (tid < a.num_seqs) {
    const int ntq = (n + kRows - 1) / kRows;
    const int off = base + incl - np;
    for (int k = 0; k < np; ++k) {
      int w = -1;  // an invalid sequence's unit goes last
      if (!bad) {
        const int rA = min((2 * k + 1) * kRows, n), rB = min((2 * k + 2) * kRows, n);
        w = (first + rA + kKeys - 1) / kKeys + (2 * k + 1 < ntq ? (first + rB + kKeys - 1) / kKeys : 0);
      }
      s_work[off + k] = w;
      s_seq[off + k] = tid;
      s_pair[off + k] = k;
    }
  }
  __syncthreads();
  for (int u = tid; u < units; u += blockDim.x) {
    int r = 0;
    const int wu = s_work[u];
    for (int v = 0; v < units; ++v) {
      const int wv = s_work[v];
      r += (wv > wu) || (wv == wu && v < u);
    }
    if (r == rank) {
      s_pick[0] = s_seq[u];
      s_pick[1] = s_pair[u];
    }
  }
  __syncthreads();
  const int seq = s_pick[0];
  *pair_out = s_pick[1];
  __syncthreads();  // the scratch is reused by the caller
  return seq;
}

// E4M3 caches: the TMA ring holds 8-bit tiles (K then V, 64 rows x 128 bytes
// each) and a converter warp widens each tile (exactly) into one of two
// 16-bit K/V buffers laid out as the 16-bit ring's stages.
constexpr int kStages8 = 4;
constexpr int kStage8Bytes = 2 * kKeys * 128;

template <typename KV>
constexpr int smem_bytes() {
  return std::is_same<KV, E4M3>::value
             ? 2 * kQBytes + kStages8 * kStage8Bytes + 2 * kStageBytes + 512 + 1024
             : 2 * kQBytes + kStages * kStageBytes + 512 + 1024;
}

template <typename KV>
constexpr int threads() {
  return std::is_same<KV, E4M3>::value ? kThreadsU + 64 : kThreadsU;  // + two converter warps
}

template <typename KV, typename Q, int T, bool kCasc = false>
__global__ void __launch_bounds__(threads<KV>(), 1)
    prefill_umma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  constexpr int D = 128;
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  constexpr bool kBf = std::is_same<KV, BF16>::value;   // MMA type: bf16, else f16
  constexpr bool kOutBf = std::is_same<Q, BF16>::value;
  constexpr int BPT = kKeys / T;   // blocks per key tile
  constexpr uint32_t kIdQK = idesc(kBf, kRows, kKeys, false);
  constexpr uint32_t kIdPV = idesc(kBf, kRows, D, true);
  constexpr int kProd = 8, kMma = 9, kConv = 10;  // warps (E4M3: converters 10 (K) and 11 (V))
  constexpr int kNS = kFp8 ? kStages8 : kStages;  // TMA ring stages
  constexpr int kNT = threads<KV>();

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the shared-prefix pass: the decode kernel behind it may start now (it
  // reads this grid's partials only after its own wait)
  if constexpr (kCasc) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid: (query head, unit rank) with the units ranked longest first, or
  // (pair counted from the chunk's end, query head, sequence); shared-prefix
  // pass: (row pair, key range, KV head)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  int j, s, qp_rev, kbeg = 0, seq0 = 0;
  if constexpr (kCasc) {
    j = blockIdx.z * a.group;   // first query head of the KV head
    s = 0;                      // the shared blocks are read through table row 0
    qp_rev = -1;                // one pair of query tiles: rows seq * G + head of this CTA's sequences
    kbeg = blockIdx.y * a.sp_split;
    seq0 = blockIdx.x * a.sp_seqs;
  } else if (a.ranked) {
    int pair = 0;
    j = blockIdx.x;
    s = ranked_unit<T>(a, blockIdx.y, reinterpret_cast<int*>(smem), &pair);
    if (s < 0) return;
    qp_rev = -1 - pair;  // marks a pair index given directly
  } else {
    qp_rev = blockIdx.x;
    j = blockIdx.y;
    s = blockIdx.z;
  }
  const int HQ = a.num_q_heads;
  // keys: positions [kbeg, ctx) (prefill: 0 .. ctx - 1, causal)
  const int ctx = kCasc ? min(a.sp_tokens, kbeg + a.sp_split) : a.ctx_lens[s];
  const int q0 = kCasc ? 0 : a.query_start[s];
  const int n = kCasc ? min(a.sp_seqs, a.num_seqs - seq0) * a.group : a.query_start[s + 1] - q0;
  if (q0 < 0 || n <= 0 || q0 + n > a.total_q) return;  // no rows this CTA may write
  const int ntq = (n + kRows - 1) / kRows;       // query tiles of the chunk
  const int npairs = (ntq + 1) / 2;
  const bool bad_len = !kCasc && (ctx < 0 || ctx > a.max_blocks * T || n > ctx || npairs > a.max_q_tiles);
  if (bad_len) {  // invalid lengths: the chunk's rows of head j become NaN
    if (tid == 0 && a.status != nullptr) atomicOr(a.status, kBadLength);
    if (qp_rev == 0 || qp_rev == -1)
      for (int i = tid; i < n * D; i += kNT)
        store_elem<Q>(a.out, (static_cast<size_t>(q0 + i / D) * HQ + j) * D + i % D, CUDART_NAN_F);
    return;
  }
  if (qp_rev >= npairs) return;
  const int qp = qp_rev < 0 ? -1 - qp_rev : npairs - 1 - qp_rev;
  if (qp >= npairs || ctx <= kbeg) return;
  const int first = ctx - n;                      // position of the chunk's first query
  // query tile X (0 = A, 1 = B): chunk rows r_begin[X] .. r_end[X] - 1
  const bool hasB = 2 * qp + 1 < ntq;
  int r_begin[2], r_end[2], nt[2];
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    r_begin[X] = (2 * qp + X) * kRows;
    r_end[X] = min(r_begin[X] + kRows, n);
    nt[X] = (X == 1 && !hasB) ? 0
            : kCasc ? (ctx - kbeg + kKeys - 1) / kKeys      // key tiles
                    : (first + r_end[X] + kKeys - 1) / kKeys;
  }
  const int n_tiles = max(nt[0], nt[1]);
  const int kvh = j / a.group;
  const HeadScales hs = head_scales(a.head_scales, a.num_kv_heads, kvh, a.softmax_scale, a.qk_scale,
                                    a.v_scale, 1.f, 1.f);

  uint8_t* q_s = smem;                                  // [X][2 slabs][128 rows][128 B]
  // 16-bit: [stage][K slab0, K slab1, V slab0, V slab1]; E4M3: [stage][K, V]
  // of 64 rows x 128 bytes, then the two widened 16-bit K/V buffers
  uint8_t* ring = smem + 2 * kQBytes;
  uint8_t* wide = ring + kStages8 * kStage8Bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      kFp8 ? wide + 2 * kStageBytes : ring + kStages * kStageBytes);
  uint64_t* full = bars;                 // [kNS] K/V landed (TMA)
  uint64_t* empty = bars + kNS;          // [kNS] stage free (16-bit: P V done; E4M3: widened)
  uint64_t* s_full = empty + kNS;        // [X][2] S buffer written (commit)
  uint64_t* p_full = s_full + 4;         // [X][2] P written over S by the tile's 128 softmax threads
  uint64_t* o_done = p_full + 4;         // [X][2] P V of a key tile done (commit)
  uint64_t* fin = o_done + 4;            // every UMMA done (commit)
  uint64_t* conv_full = fin + 1;         // E4M3: [2] widened buffer ready
  uint64_t* wide_free = conv_full + 2;   // E4M3: [2] every UMMA reading the widened buffer done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wide_free + 2);
  __shared__ int s_bad;      // PKV_DEVICE_* bits (atomicOr: several warps may set them)
  __shared__ int s_issued;   // key tiles the producer has issued
  __shared__ uint8_t s_pbad[kCasc ? 256 : 1];  // shared-prefix pass: sequence breaks the declaration

  if (tid == 0) {
    s_bad = 0;
    s_issued = 0;
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kFp8 ? 2 : 1);  // E4M3: both converter warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&conv_full[i]), 2);
      mbar_init(smem_u32(&wide_free[i]), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&p_full[i]), kRows);
      mbar_init(smem_u32(&o_done[i]), 1);
    }
    mbar_init(smem_u32(fin), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kProd) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }

  // Q rows (softmax threads of tile X): row r = chunk row r_begin[X] + r, zero
  // past the chunk's end, 128-byte-swizzled into two slabs
  if (warp < 8) {
    const int X = warp >> 2, r = tid & 127;
    const int cr = r_begin[X] + r;
    const bool in = cr < n && (X == 0 || hasB);
    // query row: chunk row cr of head j, or (shared-prefix pass) head
    // j + cr % G of sequence seq0 + cr / G
    const size_t qrow = kCasc ? static_cast<size_t>(seq0 + cr / a.group) * HQ + j + cr % a.group
                              : static_cast<size_t>(q0 + cr) * HQ + j;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const typename Q::raw*>(a.q) +
                                                      qrow * D);
    uint8_t* qx = q_s + X * kQBytes;
    // all 16 loads first (one round trip), then the shared-memory stores
    uint4 qv[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) qv[c] = in ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint4 v = qv[c];
      if constexpr (kFp8 && kOutBf) {  // the MMA is f16 (the widened E4M3): q to f16
        float f[8];
        LoadF32<Q, 8>::run(reinterpret_cast<const typename Q::raw*>(&v), f);
        v = make_uint4(pack2<false>(f[0], f[1]), pack2<false>(f[2], f[3]), pack2<false>(f[4], f[5]),
                       pack2<false>(f[6], f[7]));
      }
      *reinterpret_cast<uint4*>(qx + (c >> 3) * (kRows * 128) + sw(r, c & 7)) = v;
    }
    fence_proxy_async();
  }
  if constexpr (kCasc) {
    // the first key range of each KV head checks that its sequences' tables
    // start with the shared blocks (row 0's, which this pass reads for all)
    const int nseq = n / a.group, nb = a.sp_tokens / T;
    for (int i = tid; i < nseq; i += kNT) s_pbad[i] = 0;
    __syncthreads();
    if (blockIdx.y == 0) {
      // kU entries (and row 0's matching ones) in flight per thread
      constexpr int kU = 8;
      const int total = nseq * nb;
      for (int e0 = tid; e0 < total; e0 += kU * kNT) {
        int mine[kU], ref[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int e = e0 + u * kNT;
          mine[u] = ref[u] = 0;
          if (e < total) {
            mine[u] = __ldg(a.tables + static_cast<size_t>(seq0 + e / nb) * a.max_blocks + e % nb);
            ref[u] = __ldg(a.tables + e % nb);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (e0 + u * kNT < total && mine[u] != ref[u]) s_pbad[(e0 + u * kNT) / nb] = 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int t = 0; t < n_tiles; ++t) {
        const int slot = t % kNS;
        if (t >= kNS && !mbar_wait(smem_u32(&empty[slot]), ((t / kNS) - 1) & 1, kWaitNs)) {
          atomicOr(&s_bad, kTimeout);
          break;
        }
        uint8_t* st = ring + slot * (kFp8 ? kStage8Bytes : kStageBytes);
        int ids[BPT];
        int nbox = 0;
        for (int b = 0; b < BPT; ++b) {
          const int lb = (kbeg + t * kKeys) / T + b;
          ids[b] = -1;
          if (lb * T < ctx) {
            const int id = a.tables[static_cast<size_t>(s) * a.max_blocks + lb];
            if (id < 0 || id >= a.num_blocks) atomicOr(&s_bad, kBadTable);
            else {
              ids[b] = id;
              ++nbox;
            }
          }
        }
        const uint32_t bar = smem_u32(&full[slot]);
        constexpr int kSlabs = kFp8 ? 1 : 2;  // 128-byte slabs per row
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox) * 2u * kSlabs * (T * 128));
        for (int b = 0; b < BPT; ++b) {
          if (ids[b] < 0) continue;
          const int row = (ids[b] * a.num_kv_heads + kvh) * T;
          for (int sl = 0; sl < kSlabs; ++sl) {
            const int vo = kFp8 ? kKeys * 128 : kKVBytes;  // V after K
            tma_load_2d(smem_u32(st + sl * kSlab + b * T * 128), &kmap, sl * 128, row, bar);
            tma_load_2d(smem_u32(st + vo + sl * kSlab + b * T * 128), &vmap, sl * 128, row, bar);
          }
        }
        s_issued = t + 1;
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // descriptors of the operand bases; an operand's offset (16-byte
      // units) is added to the start-address field, which never carries
      // (shared-memory addresses are below 2^18)
      // 16-bit K/V of key tile t: ring stage t % kStages, or (E4M3) the
      // widened buffer t % 2 once the converter has filled it
      uint8_t* kv16 = kFp8 ? wide : ring;
      const uint64_t q_desc = sw128_desc(smem_u32(q_s), 16, 1024);
      const uint64_t k_desc = sw128_desc(smem_u32(kv16), 16, 1024);
      const uint64_t v_desc = sw128_desc(smem_u32(kv16 + kKVBytes), kSlab, 1024);
      auto kv_of = [&](int t) { return kFp8 ? (t & 1) : t % kStages; };
      auto qk = [&](int X, int t) -> bool {  // S_t of tile X into its buffer t & 1
        const int slot = kv_of(t), b = t & 1, i = 2 * X + b;
        const bool landed = kFp8 ? mbar_wait(smem_u32(&conv_full[slot]), (t >> 1) & 1, kWaitNs)
                                 : mbar_wait(smem_u32(&full[slot]), (t / kStages) & 1, kWaitNs);
        if (!landed) return false;
        // the buffer's previous key tile (t - 2): its P has been read by P V
        if (t >= 2 && !mbar_wait(smem_u32(&o_done[i]), ((t >> 1) - 1) & 1, kWaitNs)) return false;
        tc_fence_after();
        const uint64_t qd = q_desc + ((X * kQBytes) >> 4);
        const uint64_t kd = k_desc + ((slot * kStageBytes) >> 4);
        const uint32_t d_tmem = tmem + 256 * X + 64 * b;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off_q = ((ks >> 2) * (kRows * 128) + 32 * (ks & 3)) >> 4;
          const uint32_t off_k = ((ks >> 2) * kSlab + 32 * (ks & 3)) >> 4;
          umma(d_tmem, qd + off_q, kd + off_k, kIdQK, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&s_full[i]));
        return true;
      };
      auto pv = [&](int X, int t) -> bool {  // O_X += P_t V_t
        const int b = t & 1, i = 2 * X + b;
        if (!mbar_wait(smem_u32(&p_full[i]), (t >> 1) & 1, kWaitNs)) return false;
        tc_fence_after();
        const uint64_t vd = v_desc + ((kv_of(t) * kStageBytes) >> 4);
        const uint32_t d_tmem = tmem + 256 * X + 128;
        const uint32_t p_tmem = tmem + 256 * X + 64 * b;  // 8 columns per 16 keys
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_ts(d_tmem, p_tmem + 8 * kk, vd + ((2048 * kk) >> 4), kIdPV, (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(smem_u32(&o_done[i]));
        return true;
      };
      bool ok = true;
      for (int t = 0; t < 2 && ok; ++t)
        for (int X = 0; X < 2 && ok; ++X)
          if (t < nt[X]) ok = qk(X, t);
      for (int t = 0; t < n_tiles && ok; ++t) {
        for (int X = 0; X < 2 && ok; ++X)
          if (t < nt[X]) ok = pv(X, t);
        if (!ok) break;
        // both tiles' P V of this stage done: the stage (E4M3: the widened buffer) is free
        umma_commit(smem_u32(kFp8 ? &wide_free[t & 1] : &empty[t % kStages]));
        for (int X = 0; X < 2 && ok; ++X)
          if (t + 2 < nt[X]) ok = qk(X, t + 2);
      }
      if (!ok) atomicOr(&s_bad, kTimeout);
      umma_commit(smem_u32(fin));
    }
  } else if (kFp8 && warp >= kConv) {
    // ------------------------------------------------------------ converters
    // Each 8-bit tile (K then V, 64 rows x 128 bytes, 128-byte swizzled)
    // widened to f16 into buffer t % 2 in the 16-bit layout (two 128-byte
    // slabs per row, swizzled), V rows at positions >= ctx written as zeros;
    // warp 10 widens K, warp 11 V (on two SM sub-partitions).
    // E4M3 -> f16 is exact; the scales stay in the logit scale and in O.
    const int tv = warp - kConv;
    constexpr unsigned FULL = 0xffffffffu;
    for (int t = 0; t < n_tiles; ++t) {
      const int slot = t % kStages8, w = t & 1;
      const bool ready = mbar_wait(smem_u32(&full[slot]), (t / kStages8) & 1, kWaitNs) &&
                         (t < 2 || mbar_wait(smem_u32(&wide_free[w]), ((t >> 1) - 1) & 1, kWaitNs));
      if (!__all_sync(FULL, ready)) {
        if (lane == 0) atomicOr(&s_bad, kTimeout);
        break;
      }
      const uint8_t* src = ring + slot * kStage8Bytes;
      uint8_t* dst = wide + w * kStageBytes;
      const int kb = kbeg + t * kKeys;
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int q = lane + 32 * k;               // 16-byte chunk: row, column
        const int row = q >> 3, c = q & 7;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (!(tv == 1 && kb + row >= ctx)) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + tv * (kKeys * 128) + sw(row, c));
          lo = make_uint4(e4m3x2_f16x2(x.x & 0xffffu), e4m3x2_f16x2(x.x >> 16),
                          e4m3x2_f16x2(x.y & 0xffffu), e4m3x2_f16x2(x.y >> 16));
          hi = make_uint4(e4m3x2_f16x2(x.z & 0xffffu), e4m3x2_f16x2(x.z >> 16),
                          e4m3x2_f16x2(x.w & 0xffffu), e4m3x2_f16x2(x.w >> 16));
        }
        // head_dim 16c .. 16c + 15: slab c / 4, 16-byte chunks 2 (c % 4) and 2 (c % 4) + 1
        uint8_t* d = dst + tv * kKVBytes + (c >> 2) * kSlab;
        *reinterpret_cast<uint4*>(d + sw(row, 2 * (c & 3))) = lo;
        *reinterpret_cast<uint4*>(d + sw(row, 2 * (c & 3) + 1)) = hi;
      }
      fence_proxy_async();  // the widened tile, before the tensor core reads it
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&conv_full[w]));
        mbar_arrive(smem_u32(&empty[slot]));  // the 8-bit stage may be refilled
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    // Every branch around a TMEM load or store (warp-wide, .sync.aligned)
    // is taken by the whole warp: waits are combined with __all_sync and a
    // row that moves its reference moves it inside a warp-wide rescale.
    constexpr unsigned FULL = 0xffffffffu;
    const int X = warp >> 2;                  // query tile
    const int r = tid & 127;                  // query row, TMEM lane
    const int cr = r_begin[X] + r;
    const int pos = first + cr;               // query position
    const int ntx = nt[X];
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + 256 * X + 128;
    // the logit scale the exponent applies (16-bit caches: softmax_scale * log2 e > 0)
    const float qe = (!kFp8 || hs.qk > 0.f) ? hs.qk : 1.f;
    float m_ref = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntx; ++t) {
      const int b = t & 1, i = 2 * X + b;
      if (!__all_sync(FULL, mbar_wait(smem_u32(&s_full[i]), (t >> 1) & 1, kWaitNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[64];
      {
        uint32_t h0[32], h1[32];
        const uint32_t ts = tmem + 256 * X + 64 * b + lane_off;
        tmem_ld32_async(ts, h0);
        tmem_ld32_async(ts + 32, h1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sv[e] = __uint_as_float(h0[e]);
          sv[32 + e] = __uint_as_float(h1[e]);
        }
      }

      // mask the keys after the query (and past ctx); the row maximum of the
      // raw scores in eight independent chains, scaled once (the scale is
      // positive, so it commutes with the maximum); the exponent below takes
      // s * scale - m as one fused multiply-add
      const int kb = kbeg + t * kKeys;
      const int lim = (kCasc ? ctx - 1 : min(pos, ctx - 1)) - kb;   // keys kb + e, e <= lim, attended
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = -CUDART_INF_F;
      if (lim < kKeys - 1) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e > lim) sv[e] = -CUDART_INF_F;
      }
      if constexpr (kFp8) {
        if (!(hs.qk > 0.f)) {  // an E4M3 scale <= 0 (the host sends softmax scales <= 0
#pragma unroll               // to the mma.sync kernel): scale first, then the maximum
          for (int e = 0; e < 64; ++e)
            if (sv[e] != -CUDART_INF_F) sv[e] *= hs.qk;
        }
      }
#pragma unroll
      for (int e = 0; e < 64; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], sv[e]);
      const float mx = qe * fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                  fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const bool move = mx > m_ref + kRescaleLog2;
      const bool scale = move && t > 0 && m_ref != -CUDART_INF_F;  // O holds earlier tiles
      if (__any_sync(FULL, scale)) {
        // rows that move their reference scale their row of O (every P V so
        // far done); the others multiply by 1
        const int ip = 2 * X + ((t - 1) & 1);
        if (!__all_sync(FULL, mbar_wait(smem_u32(&o_done[ip]), ((t - 1) >> 1) & 1, kWaitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = scale ? ex2(m_ref - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + lane_off + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= f;
          tmem_st32(tO + lane_off + c, o);
        }
        l *= f;
      }
      if (move) m_ref = mx;
      // P_t over the first 32 columns of the S buffer just read: column c
      // holds keys 2c, 2c + 1 (the K order of the A operand in TMEM)
      float sum8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sum8[k] = 0.f;
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(sv[2 * c], qe, -m_ref));
        const float p1 = ex2(fmaf(sv[2 * c + 1], qe, -m_ref));
        sum8[(2 * c) & 7] += p0;
        sum8[(2 * c + 1) & 7] += p1;
        w[c] = pack2<kBf>(p0, p1);
      }
      tmem_st32u(tmem + 256 * X + 64 * b + lane_off, w);
      l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      // V rows at positions >= ctx (the tail of the last block, blocks not
      // loaded) are zeroed by tile A's threads (tile B's too when A has no
      // such tile): 64 rows of 2 x 128 bytes, one row per thread
      if (!kFp8 && kb + kKeys > ctx && r < kKeys && kb + r >= ctx && (X == 0 || t >= nt[0])) {
        uint8_t* vt = ring + (t % kStages) * kStageBytes + kKVBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vt + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vt + kSlab + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();  // before the tensor core reads V
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&p_full[i]));
    }
    // epilogue: O / l of the row, after the tile's last P V (shared-prefix
    // pass: the row's partial m_ref, l and O times the V scale)
    if (ntx > 0) {
      const int tl = ntx - 1;
      ok = __all_sync(FULL, ok && mbar_wait(smem_u32(&o_done[2 * X + (tl & 1)]), (tl >> 1) & 1, kWaitNs));
      tc_fence_after();
      if (!ok) atomicOr(&s_bad, kTimeout);
      const bool row_in = cr < r_end[X];
      bool bad = !ok || *reinterpret_cast<volatile int*>(&s_bad) != 0;
      if constexpr (kCasc) {
        if (row_in && s_pbad[cr / a.group]) {
          bad = true;
          if (a.status != nullptr) atomicOr(a.status, kBadPrefix);
        }
      }
      if constexpr (kCasc) {
        const size_t pidx = (static_cast<size_t>(seq0 + cr / a.group) * HQ + j + cr % a.group) *
                                a.max_splits + a.sp_slot0 + blockIdx.y;
        float* acc = a.ws_acc + pidx * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + lane_off + c, o);
          if (row_in) {
            float4* d4 = reinterpret_cast<float4*>(acc + c);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = bad ? make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F)
                          : make_float4(o[4 * e] * hs.v, o[4 * e + 1] * hs.v, o[4 * e + 2] * hs.v,
                                        o[4 * e + 3] * hs.v);
          }
        }
        if (row_in) {
          a.ws_m[pidx] = m_ref;
          a.ws_l[pidx] = bad ? CUDART_NAN_F : l;
        }
      } else {
        const float inv = (l > 0.f || l != l) ? hs.v / l : 0.f;
        typename Q::raw* dst =
            static_cast<typename Q::raw*>(a.out) + (static_cast<size_t>(q0 + cr) * HQ + j) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + lane_off + c, o);
          if (row_in) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack2<kOutBf>(bad ? CUDART_NAN_F : o[2 * e] * inv,
                                   bad ? CUDART_NAN_F : o[2 * e + 1] * inv);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- exit
  // every UMMA done and every copy landed before TMEM and shared memory go
  __syncthreads();
  if (tid == 0) {
    mbar_wait(smem_u32(fin), 0, kDrainNs);
    if (s_bad) {
      // the copies of the last tiles issued may still be landing
      const int issued = s_issued;
      for (int t = max(0, issued - kNS); t < issued; ++t)
        mbar_wait(smem_u32(&full[t % kNS]), (t / kNS) & 1, kDrainNs);
      if (a.status != nullptr) atomicOr(a.status, s_bad);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProd) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace umma
}  // namespace tc
}  // namespace pkv
