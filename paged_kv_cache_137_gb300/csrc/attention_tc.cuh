// Tensor-core paged decode attention with TMA-staged K/V tiles.
//
// What it computes is the same as the CUDA-core kernel (attention_simt.cuh):
// for the G query heads of one KV head, softmax(q . K^T * scale) V over the
// logical positions of one split, K/V gathered through the block table (the
// katajob Q&A, "The paging idea"; the foundry page on paged block allocation,
// "Concept").
//
// How, on GB300:
//  * One CTA per (KV head, sequence, split): four warps and 64-token tiles by
//    default; behind a shared-prefix pass, where the contexts left are short,
//    one warp (block size 16) or two (block size 32) with 16- or 32-token
//    tiles, so that more CTAs per SM overlap each one's fixed latencies (at
//    block size 16 the tail queue of attention_tail.cuh runs instead where
//    its unit list fits).  The
//    split's block ids are read into shared memory; split 0 fetches its first
//    tiles' ids and its query rows together with the length.  Warp 0 refills
//    a ring of NS stages, one lane per TMA box: each stage is a tile of K and
//    of V, one box per (block, K|V) carrying the block's T rows of the head,
//    at row (block * N_kv + head) * T of the pool viewed as [rows][row_bytes]
//    (a 3-D (128 bytes, slab, row) view for 256-byte rows, so one box carries
//    both slabs), with the hardware 128-byte swizzle so that ldmatrix reads
//    are conflict-free.  Completion is tracked by one mbarrier per stage
//    (expect-tx bytes).
//  * Each warp owns 16 tokens of a tile.  Groups of up to 8 query heads take
//    the head-columns form: S^T = K q^T and O^T += V^T P^T by m16n8k16 MMAs
//    with the tokens (then head_dim) as the 16 MMA rows and the heads as the
//    8 columns, P^T reaching the B operand through movmatrix; larger groups
//    (up to 16) the head-rows form (q K^T with the heads as M).  The online
//    softmax runs on the accumulator fragments in the log2 domain.  16-bit
//    caches use bf16/f16 MMAs; an E4M3 cache is widened to f16 in registers
//    (exact) and q is converted to f16.
//  * Tokens past the context end are masked to -inf, and their V rows are
//    zeroed in shared memory before the P V MMA (0 * NaN would poison it).
//  * The warps' (max, sum, output) are merged through shared memory.  A
//    pair's tiles are shared out evenly over its splits.  With several
//    splits each CTA writes its partial and the last of the (sequence, KV
//    head)'s splits to arrive (an atomic counter, no waiting) gathers them
//    all into shared memory, merges them and resets the counter.  Behind a
//    shared-prefix pass the CTAs only write their partials; a merge kernel
//    after this one combines them with the pass's.
//  * The step's new token can be written by the CTA that holds position
//    ctx - 1, before any copy is issued (the fused slot write).
//  * Every mbarrier wait is bounded; a stage wait that gives up (its limit is
//    pkv_set_stage_wait_limit's) turns the heads' output into NaN and sets a
//    bit in the device error word, after waiting (with its own bound) for the
//    copies still in flight.
#pragma once

#include <cuda.h>
#include <math_constants.h>

#include <type_traits>

#include "attention.h"
#include "device_common.cuh"

namespace pkv {
namespace tc {

constexpr int kWarps = 4;                 // warps of the split kernel's CTA (or 2: see below)
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 64;                 // tokens per stage, 16 per warp
constexpr int kMaxTableEntries = 1024;    // block ids of one split kept in shared memory
// The narrow forms (16-bit head_dim-128 caches behind a shared-prefix pass,
// where the contexts left are short): one warp per CTA with 16-token stages of
// 8 KiB, eleven CTAs per SM (block size 16), or two warps with 32-token
// stages of 16 KiB, six CTAs per SM (block size 32); at most 512 block ids a
// split.
constexpr int kMaxTableEntries2 = 512;
template <int W>
constexpr int max_table_entries() { return W <= 2 ? kMaxTableEntries2 : kMaxTableEntries; }

constexpr uint64_t kWaitNs = 50000000ull;  // a stage wait gives up after 50 ms
constexpr uint64_t kDrainNs = 10000000ull; // after a give-up, 10 ms per copy in flight

template <typename KV, int D, int W = kWarps>
struct Geom {
  static constexpr int kElemBytes = KV::bytes;
  static constexpr int kRowBytes = D * kElemBytes;
  static constexpr int kSlabs = kRowBytes / 128;  // 128-byte column slabs per row (1 or 2)
  static constexpr int kTileBytes = 16 * W * kRowBytes;  // 16 tokens per warp
  static constexpr int kStageBytes = 2 * kTileBytes;  // K and V
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte slabs");
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false if the phase did not complete within limit_ns (or
// 2^26 attempts, whichever comes first).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;  // the common case reads no timer
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// A decode stage wait: bounded by limit_ns; a limit of 0 gives up at once
// (the failure path, exercised on purpose).
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return limit_ns != 0 && mbar_wait(bar, parity, limit_ns);
}

// Device error bits (the PKV_DEVICE_* values of the C ABI).
constexpr int kBadLength = PKV_DEVICE_BAD_LENGTH;
constexpr int kBadTable = PKV_DEVICE_BAD_TABLE;
constexpr int kTimeout = PKV_DEVICE_WAIT_TIMEOUT;
constexpr int kBadPrefix = PKV_DEVICE_BAD_SHARED_PREFIX;

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool BF>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(d) : "r"(a), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two_bytes)));
  return r;
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Byte offset of 16-byte chunk c of tile row r under the 128-byte swizzle.
// A tile stores its rows back to back, each as S 128-byte lines (one per
// 128-byte slab of the row, the order a TMA box over (bytes, slab, row)
// writes them), and the swizzle XORs a chunk's index with its line's index
// mod 8 (the tile base is 1024-byte aligned).
template <int S>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  const int line = r * S + (c >> 3);
  return static_cast<uint32_t>((line << 7) + (((c & 7) ^ (line & 7)) << 4));
}

// One TMA box of a (block, KV head): its T rows, all slabs of each row (a 2-D
// map for 128-byte rows, a 3-D (bytes, slab, row) map for 256-byte rows).
template <typename KV, int D>
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int row, uint32_t bar) {
  if constexpr (Geom<KV, D>::kSlabs == 1) tma_load_2d(dst, map, 0, row, bar);
  else tma_load_3d(dst, map, 0, 0, row, bar);
}

// ------------------------------------------------------- tile building blocks
// One warp's online-softmax state for up to 16 query heads (rows g, g + 8).
template <int D>
struct WarpState {
  float o[D / 8][4];
  float m[2], l[2];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = -CUDART_INF_F;
    l[0] = l[1] = 0.f;
  }
};

// q fragments (A operand of q . K^T) of the G heads stored row-major at qrows
// (global or shared memory); rows >= G are zero.  For an E4M3 cache q becomes
// f16 with head_dim permuted within each 16-element step so that one 32-bit
// K load of 4 bytes serves both halves of the k-step.
template <typename KV, typename Q, int D>
__device__ __forceinline__ void load_q(uint32_t (&qa)[D / 16][4], const typename Q::raw* qrows,
                                       int G, int g, int q4) {
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = g + 8 * h;
      uint32_t lo = 0, hi = 0;
      if (row < G) {
        if constexpr (!kFp8) {
          const uint32_t* qp = reinterpret_cast<const uint32_t*>(qrows + row * D + 16 * ks + 2 * q4);
          lo = qp[0];
          hi = qp[4];
        } else {
          float f[4];
          LoadF32<Q, 4>::run(qrows + row * D + 16 * ks + 4 * q4, f);
          lo = pack2<false>(f[0], f[1]);
          hi = pack2<false>(f[2], f[3]);
        }
      }
      qa[ks][h] = lo;      // a0 (row g) / a1 (row g + 8)
      qa[ks][2 + h] = hi;  // a2 / a3
    }
}

// Column of head_dim held by fragment column j of p . V n-tile n.
template <bool kFp8>
__device__ __forceinline__ int out_col(int n, int j, int q4) {
  if constexpr (!kFp8) return 8 * n + 2 * q4 + j;
  else return 16 * (n >> 1) + 4 * q4 + 2 * j + (n & 1);
}

// One warp's 16 tokens (tile rows row0 .. row0 + 15, nvalid of them inside
// the context) folded into its state.  kt/vt: the stage's K and V tiles.
// Returns true if V rows were zeroed (generic writes the caller must fence
// before the slot is refilled by TMA).
template <typename KV, int D>
__device__ __forceinline__ bool tile_step(WarpState<D>& st, const uint32_t (&qa)[D / 16][4],
                                          const uint8_t* kt, uint8_t* vt, int row0, int nvalid,
                                          float qk_scale, int lane) {
  using G_ = Geom<KV, D>;
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  constexpr bool kBf = std::is_same<KV, BF16>::value;
  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  const int q4 = lane & 3;
  bool zeroed = false;
  if (nvalid < 16) {  // zero the V rows past the context end
    const int nz = (16 - nvalid) * G_::kSlabs * 8;
    for (int i = lane; i < nz; i += 32) {
      const int r = row0 + nvalid + i / (G_::kSlabs * 8);
      const int c = i % (G_::kSlabs * 8);
      *reinterpret_cast<uint4*>(vt + swz<G_::kSlabs>(r, c)) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    zeroed = true;
  }
  const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
  const int li = lane & 7, mi = lane >> 3;

  // S = q . K^T : two n-tiles of 8 tokens
  float sc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const int r = row0 + 8 * nt + li;
    if constexpr (!kFp8) {
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz<G_::kSlabs>(r, 2 * ks + mi), b0, b1, b2, b3);
        mma16816<kBf>(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma16816<kBf>(sc[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
      }
    } else {
#pragma unroll
      for (int c0 = 0; c0 < KS; c0 += 4) {
        uint32_t w[4];
        ldsm_x4(kbase + swz<G_::kSlabs>(r, c0 + mi), w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ks = c0 + j;
          mma16816<false>(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3],
                          e4m3x2_f16x2(w[j] & 0xffffu), e4m3x2_f16x2(w[j] >> 16));
        }
      }
    }
  }

  // online softmax on the fragments: rows g (h = 0) and g + 8 (h = 1)
  float p[2][4];
  float corr[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 8 * nt + 2 * q4 + j;
        float v = sc[nt][2 * h + j] * qk_scale;
        v = col < nvalid ? v : -CUDART_INF_F;
        sc[nt][2 * h + j] = v;
        mx = fmaxf(mx, v);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(st.m[h], mx);
    corr[h] = exp2f(st.m[h] - mn);
    st.m[h] = mn;
    float sum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float e = exp2f(sc[nt][2 * h + j] - mn);
        p[nt][2 * h + j] = e;
        sum += e;
      }
    st.l[h] = st.l[h] * corr[h] + sum;
  }
  // a row whose maximum did not grow has corr exactly 1: the rescale is
  // skipped when that holds for every row of the warp (the result is the same)
  if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      st.o[n][0] *= corr[0];
      st.o[n][1] *= corr[0];
      st.o[n][2] *= corr[1];
      st.o[n][3] *= corr[1];
    }
  }
  const uint32_t pa0 = pack2<kBf>(p[0][0], p[0][1]);
  const uint32_t pa1 = pack2<kBf>(p[0][2], p[0][3]);
  const uint32_t pa2 = pack2<kBf>(p[1][0], p[1][1]);
  const uint32_t pa3 = pack2<kBf>(p[1][2], p[1][3]);

  // O += P . V
  const int rv = row0 + (mi & 1) * 8 + li;
  if constexpr (!kFp8) {
#pragma unroll
    for (int c = 0; c < NT; c += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbase + swz<G_::kSlabs>(rv, c + (mi >> 1)), b0, b1, b2, b3);
      mma16816<kBf>(st.o[c], pa0, pa1, pa2, pa3, b0, b1);
      mma16816<kBf>(st.o[c + 1], pa0, pa1, pa2, pa3, b2, b3);
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 16; c += 2) {
      uint32_t w0, w1, w2, w3;  // (tok 0-7, c), (tok 8-15, c), (0-7, c+1), (8-15, c+1)
      ldsm_x4_t(vbase + swz<G_::kSlabs>(rv, c + (mi >> 1)), w0, w1, w2, w3);
      const uint32_t x0 = prmt(w0, 0x3120), x1 = prmt(w1, 0x3120);
      const uint32_t x2 = prmt(w2, 0x3120), x3 = prmt(w3, 0x3120);
      // chunk c: even d -> n-tile 2c, odd d -> 2c + 1
      mma16816<false>(st.o[2 * c], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x0 & 0xffffu),
                      e4m3x2_f16x2(x1 & 0xffffu));
      mma16816<false>(st.o[2 * c + 1], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x0 >> 16),
                      e4m3x2_f16x2(x1 >> 16));
      mma16816<false>(st.o[2 * c + 2], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x2 & 0xffffu),
                      e4m3x2_f16x2(x3 & 0xffffu));
      mma16816<false>(st.o[2 * c + 3], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x2 >> 16),
                      e4m3x2_f16x2(x3 >> 16));
    }
  }
  return zeroed;
}

// Publish one warp's state to the merge buffers: mS/lS [warp][16] (all 16
// rows), oS [warp][ostride rows][D] (rows < G).  The sums are completed across
// the quad first.
template <typename KV, int D>
__device__ __forceinline__ void publish(const WarpState<D>& st, float* mS, float* lS, float* oS,
                                        int warp, int G, int ostride, int lane) {
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = st.l[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (q4 == 0) {
      mS[warp * 16 + g + 8 * h] = st.m[h];
      lS[warp * 16 + g + 8 * h] = l;
    }
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int d = out_col<kFp8>(n, j, q4);
      if (g < G) oS[(warp * ostride + g) * D + d] = st.o[n][j];
      if (g + 8 < G) oS[(warp * ostride + g + 8) * D + d] = st.o[n][2 + j];
    }
}

// ---------------------------------- head-columns form (query group <= 8)
// With at most 8 query heads per KV head the products run with the tokens as
// the MMA rows: S^T = K q^T (m16n8k16: 16 tokens x 8 heads, k = head_dim) and
// O^T += V^T P^T (16 head_dim rows x 8 heads, k = 16 tokens).  No MMA row is
// padding, so a warp issues half the MMAs of the head-rows form and keeps
// half the accumulators (32 instead of 64 at head_dim 128); P^T reaches the
// B operand of the second product through a warp transpose (movmatrix).
// Lane (g, q4) holds heads 2 q4 and 2 q4 + 1.

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <int D>
struct WarpStateT {
  float o[D / 16][4];  // O^T m-tile mt: (row g, head 2q4), (g, 2q4 + 1), (g + 8, 2q4), (g + 8, 2q4 + 1)
  float m[2], l[2];    // heads 2 q4 + j
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int n = 0; n < D / 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = -CUDART_INF_F;
    l[0] = l[1] = 0.f;
  }
};

// q as the B operand of S^T = K q^T: for k-step ks lane (g, q4) holds head
// g's elements k = 2 q4, 2 q4 + 1 (qb[ks][0]) and 2 q4 + 8, 2 q4 + 9
// (qb[ks][1]); heads >= G are zero.  For an E4M3 cache q becomes f16 and the
// k order within a 16-element step is the one the K bytes arrive in: lane q4
// holds head_dim 4 q4 .. 4 q4 + 3 of the step.
template <typename KV, typename Q, int D>
__device__ __forceinline__ void load_qt(uint32_t (&qb)[D / 16][2], const typename Q::raw* qrows,
                                        int G, int g, int q4) {
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t lo = 0, hi = 0;
    if (g < G) {
      if constexpr (!kFp8) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(qrows + g * D + 16 * ks + 2 * q4);
        lo = qp[0];
        hi = qp[4];
      } else {
        float f[4];
        LoadF32<Q, 4>::run(qrows + g * D + 16 * ks + 4 * q4, f);
        lo = pack2<false>(f[0], f[1]);
        hi = pack2<false>(f[2], f[3]);
      }
    }
    qb[ks][0] = lo;
    qb[ks][1] = hi;
  }
}

// head_dim held by O^T m-tile mt, fragment row g (+ 8 when hi).  E4M3 V
// arrives as byte pairs (d, d + 1) of one token: rows g and g + 8 of an
// m-tile hold d = 16 mt + 2 g and 16 mt + 2 g + 1.
template <bool kFp8>
__device__ __forceinline__ int out_row_t(int mt, int g, int hi) {
  if constexpr (!kFp8) return 16 * mt + g + 8 * hi;
  else return 16 * mt + 2 * g + hi;
}

// tile_step in the head-columns form (same contract).
template <typename KV, int D>
__device__ __forceinline__ bool tile_step_t(WarpStateT<D>& st, const uint32_t (&qb)[D / 16][2],
                                            const uint8_t* kt, uint8_t* vt, int row0, int nvalid,
                                            float qk_scale, int lane) {
  using G_ = Geom<KV, D>;
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  constexpr bool kBf = std::is_same<KV, BF16>::value;
  constexpr int KS = D / 16;
  constexpr int MT = D / 16;
  const int g = lane >> 2;
  bool zeroed = false;
  if (nvalid < 16) {  // zero the V rows past the context end
    const int nz = (16 - nvalid) * G_::kSlabs * 8;
    for (int i = lane; i < nz; i += 32) {
      const int r = row0 + nvalid + i / (G_::kSlabs * 8);
      const int c = i % (G_::kSlabs * 8);
      *reinterpret_cast<uint4*>(vt + swz<G_::kSlabs>(r, c)) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    zeroed = true;
  }
  const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
  const int li = lane & 7, mi = lane >> 3;

  // S^T = K q^T: 16 tokens x 8 heads
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (!kFp8) {
    // matrix mi: tokens (mi & 1) * 8 .., 16-byte chunk 2 ks + (mi >> 1)
    const int r = row0 + (mi & 1) * 8 + li;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kbase + swz<G_::kSlabs>(r, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
      mma16816<kBf>(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
    }
  } else {
    // matrix mi: tokens (mi & 1) * 8 .., 16-byte chunk ks + (mi >> 1): one
    // load serves two k-steps; a register holds head_dim 4 q4 .. 4 q4 + 3
    const int r = row0 + (mi & 1) * 8 + li;
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
      uint32_t w0, w1, w2, w3;
      ldsm_x4(kbase + swz<G_::kSlabs>(r, ks + (mi >> 1)), w0, w1, w2, w3);
      mma16816<false>(sc, e4m3x2_f16x2(w0 & 0xffffu), e4m3x2_f16x2(w1 & 0xffffu),
                      e4m3x2_f16x2(w0 >> 16), e4m3x2_f16x2(w1 >> 16), qb[ks][0], qb[ks][1]);
      mma16816<false>(sc, e4m3x2_f16x2(w2 & 0xffffu), e4m3x2_f16x2(w3 & 0xffffu),
                      e4m3x2_f16x2(w2 >> 16), e4m3x2_f16x2(w3 >> 16), qb[ks + 1][0],
                      qb[ks + 1][1]);
    }
  }

  // online softmax over the tokens (rows g, g + 8) of heads 2 q4 + j
  float p[4];
  float corr[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float v0 = g < nvalid ? sc[j] * qk_scale : -CUDART_INF_F;
    const float v1 = g + 8 < nvalid ? sc[2 + j] * qk_scale : -CUDART_INF_F;
    float mx = fmaxf(v0, v1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(st.m[j], mx);
    corr[j] = exp2f(st.m[j] - mn);
    st.m[j] = mn;
    p[j] = exp2f(v0 - mn);
    p[2 + j] = exp2f(v1 - mn);
    st.l[j] = st.l[j] * corr[j] + (p[j] + p[2 + j]);
  }
  // a head whose maximum did not grow has corr exactly 1: the rescale is
  // skipped when that holds for every head of the warp (the result is the same)
  if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      st.o[mt][0] *= corr[0];
      st.o[mt][1] *= corr[1];
      st.o[mt][2] *= corr[0];
      st.o[mt][3] *= corr[1];
    }
  }
  // P^T as the B operand (k = tokens, n = heads): the transposes of the
  // (tokens 0-7) x heads and (tokens 8-15) x heads blocks
  const uint32_t pb0 = movmatrix_t(pack2<kBf>(p[0], p[1]));
  const uint32_t pb1 = movmatrix_t(pack2<kBf>(p[2], p[3]));

  // O^T += V^T P^T
  if constexpr (!kFp8) {
    // matrix mi: tokens (mi >> 1) * 8 .., 16-byte chunk 2 mt + (mi & 1)
    const int rv = row0 + (mi >> 1) * 8 + li;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vbase + swz<G_::kSlabs>(rv, 2 * mt + (mi & 1)), a0, a1, a2, a3);
      mma16816<kBf>(st.o[mt], a0, a1, a2, a3, pb0, pb1);
    }
  } else {
    // matrix mi: tokens (mi & 1) * 8 .., 16-byte chunk mt + (mi >> 1); a
    // register holds tokens 2 q4, 2 q4 + 1 of head_dim pair (2 g, 2 g + 1)
    const int rv = row0 + (mi & 1) * 8 + li;
#pragma unroll
    for (int mt = 0; mt < MT; mt += 2) {
      uint32_t w0, w1, w2, w3;  // (tok 0-7, mt), (tok 8-15, mt), (0-7, mt+1), (8-15, mt+1)
      ldsm_x4_t(vbase + swz<G_::kSlabs>(rv, mt + (mi >> 1)), w0, w1, w2, w3);
      const uint32_t x0 = prmt(w0, 0x3120), x1 = prmt(w1, 0x3120);
      const uint32_t x2 = prmt(w2, 0x3120), x3 = prmt(w3, 0x3120);
      mma16816<false>(st.o[mt], e4m3x2_f16x2(x0 & 0xffffu), e4m3x2_f16x2(x0 >> 16),
                      e4m3x2_f16x2(x1 & 0xffffu), e4m3x2_f16x2(x1 >> 16), pb0, pb1);
      mma16816<false>(st.o[mt + 1], e4m3x2_f16x2(x2 & 0xffffu), e4m3x2_f16x2(x2 >> 16),
                      e4m3x2_f16x2(x3 & 0xffffu), e4m3x2_f16x2(x3 >> 16), pb0, pb1);
    }
  }
  return zeroed;
}

// publish in the head-columns form: mS/lS [warp][16] (heads < 8), oS
// [warp][ostride][D] (heads < G).  The sums are completed across the eight
// token rows first.
template <typename KV, int D>
__device__ __forceinline__ void publish_t(const WarpStateT<D>& st, float* mS, float* lS, float* oS,
                                          int warp, int G, int ostride, int lane) {
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = st.l[j];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (g == 0) {
      mS[warp * 16 + 2 * q4 + j] = st.m[j];
      lS[warp * 16 + 2 * q4 + j] = l;
    }
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int head = 2 * q4 + (e & 1);
      if (head < G) oS[(warp * ostride + head) * D + out_row_t<kFp8>(mt, g, e >> 1)] = st.o[mt][e];
    }
}

// Combine nw published states for row `row`, column d:
// M = max m_w, L = sum l_w 2^(m_w - M), A = sum o_w 2^(m_w - M).
__device__ __forceinline__ void combine_warps(const float* mS, const float* lS, const float* oS,
                                              int nw, int ostride, int row, int d, int D, float& M,
                                              float& L, float& A) {
  M = -CUDART_INF_F;
  for (int w = 0; w < nw; ++w) M = fmaxf(M, mS[w * 16 + row]);
  L = 0.f;
  A = 0.f;
  if (M != -CUDART_INF_F) {
    for (int w = 0; w < nw; ++w) {
      const float f = exp2f(mS[w * 16 + row] - M);
      L = fmaf(lS[w * 16 + row], f, L);
      A = fmaf(oS[(w * ostride + row) * D + d], f, A);
    }
  }
}

// Whether the partials of nsplit split slots of a query group fit the
// shared-memory gather below (`cap` floats, NT threads).
template <int D, int NT>
__device__ __forceinline__ bool gather_fits(int G, int nsplit, int cap) {
  return G * nsplit <= NT && G * nsplit * (D + 2) <= cap;
}

// Gather the partials (m, l, a) of the G heads at head0 from the split slots
// slot(0) .. slot(nsplit - 1) into shared memory: a [G][nsplit][D], then m
// and l [G][nsplit].  Every load is a global round trip of several
// microseconds while the GPU streams, so they are all issued before any is
// used.  Ends with a CTA barrier.
template <int D, int NT, typename Slot>
__device__ void gather_partials(const DecodeArgs& a, size_t head0, int nsplit, Slot slot,
                                float* stage) {
  const int tid = threadIdx.x, G = a.group;
  const int nacc = G * nsplit * D;
  float* g_acc = stage;
  float* g_m = g_acc + nacc;
  float* g_l = g_m + G * nsplit;
  float mv = 0.f, lv = 0.f;
  if (tid < G * nsplit) {
    const size_t pidx = (head0 + tid / nsplit) * a.max_splits + slot(tid % nsplit);
    mv = __ldcg(a.ws_m + pidx);
    lv = __ldcg(a.ws_l + pidx);
  }
  constexpr int kU = 8;  // float4 loads in flight per thread
  for (int i0 = 0; i0 < nacc / 4; i0 += kU * NT) {
    float4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * NT + tid;
      if (i < nacc / 4) {
        const int e = 4 * i, row = e / (nsplit * D), rem = e - row * nsplit * D;
        const int sp = rem / D, d = rem - sp * D;
        v[u] = __ldcg(reinterpret_cast<const float4*>(
            a.ws_acc + ((head0 + row) * a.max_splits + slot(sp)) * D + d));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * NT + tid;
      if (i < nacc / 4) reinterpret_cast<float4*>(g_acc)[i] = v[u];
    }
  }
  if (tid < G * nsplit) {
    g_m[tid] = mv;
    g_l[tid] = lv;
  }
  __syncthreads();
}

// Combine the partials (max m_i, sum l_i, unnormalised output a_i) of the G
// heads at head0, from split slots 0 .. nsplit - 1 and extra_base ..
// extra_base + n_extra - 1:  M = max m_i, L = sum l_i 2^(m_i - M),
// o = sum a_i 2^(m_i - M) / L.  The partials are gathered into shared
// memory (stage, `cap` floats) first where they fit.
template <typename Q, int D, int NT>
__device__ void merge_splits(const DecodeArgs& a, size_t head0, int nsplit_tail, int extra_base,
                             int n_extra, float* stage, int cap) {
  const int tid = threadIdx.x, G = a.group;
  const int nsplit = nsplit_tail + n_extra;   // partials in all
  auto slot = [&](int i) { return i < nsplit_tail ? i : extra_base + (i - nsplit_tail); };
  if (gather_fits<D, NT>(G, nsplit, cap)) {
    gather_partials<D, NT>(a, head0, nsplit, slot, stage);
    const float* g_acc = stage;
    const float* g_m = g_acc + G * nsplit * D;
    const float* g_l = g_m + G * nsplit;
    for (int i = tid; i < G * D; i += NT) {
      const int row = i / D, d = i % D;
      float M = -CUDART_INF_F;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, g_m[row * nsplit + sp]);
      float L = 0.f, A = 0.f;
      if (M != -CUDART_INF_F) {
        for (int sp = 0; sp < nsplit; ++sp) {
          const float f = exp2f(g_m[row * nsplit + sp] - M);
          L = fmaf(g_l[row * nsplit + sp], f, L);
          A = fmaf(g_acc[(row * nsplit + sp) * D + d], f, A);
        }
      } else {
        // no split attended a position: the sums are 0, or NaN for a split
        // that failed, which must reach the output
        for (int sp = 0; sp < nsplit; ++sp) L += g_l[row * nsplit + sp];
      }
      store_elem<Q>(a.out, (head0 + row) * D + d, (L > 0.f || L != L) ? A / L : 0.f);
    }
  } else {
    for (int i = tid; i < G * D; i += NT) {
      const int row = i / D, d = i % D;
      const size_t base = (head0 + row) * a.max_splits;
      float M = -CUDART_INF_F;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(a.ws_m + base + slot(sp)));
      float L = 0.f, A = 0.f;
      if (M != -CUDART_INF_F) {
        for (int sp = 0; sp < nsplit; ++sp) {
          const float f = exp2f(__ldcg(a.ws_m + base + slot(sp)) - M);
          L = fmaf(__ldcg(a.ws_l + base + slot(sp)), f, L);
          A = fmaf(__ldcg(a.ws_acc + (base + slot(sp)) * D + d), f, A);
        }
      } else {
        for (int sp = 0; sp < nsplit; ++sp) L += __ldcg(a.ws_l + base + slot(sp));
      }
      store_elem<Q>(a.out, (head0 + row) * D + d, (L > 0.f || L != L) ? A / L : 0.f);
    }
  }
}

// ------------------------------------------------------------------ kernel
// Resident CTAs per SM the split kernel is compiled for: four for the E4M3
// head-columns form (126 registers, a 48 KiB ring), three otherwise.
template <typename KV, bool HC>
constexpr int split_ctas_per_sm() {
  return HC && std::is_same<KV, E4M3>::value ? 4 : 3;
}

template <typename KV, bool HC, int W>
constexpr int resident_ctas() { return W == 1 ? 11 : W == 2 ? 6 : split_ctas_per_sm<KV, HC>(); }

// HC: the head-columns form of the tile products (query group <= 8).  W:
// warps per CTA, 16 tokens of each W * 16-token tile per warp (4; or 1 or 2,
// with more CTAs per SM, for the short contexts past a shared prefix).
template <typename KV, typename Q, int D, int T, int NS, bool HC, int W = kWarps>
__global__ void __launch_bounds__(32 * W, resident_ctas<KV, HC, W>())
    decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
  using G_ = Geom<KV, D, W>;
  constexpr int kWarps = W, kThreads = 32 * W, kTile = 16 * W;
  constexpr int kMaxTableEntries = max_table_entries<W>();
  using State = std::conditional_t<HC, WarpStateT<D>, WarpState<D>>;
  constexpr int KS = D / 16;        // k-steps of q . K^T
  constexpr int BPT = kTile / T;    // blocks per tile
  constexpr int kBoxBytes = T * G_::kRowBytes;  // one (block, head) box: all its slabs
  static_assert(kTile % T == 0, "a tile holds whole blocks");

  // split-major grid: every pair's first split is dispatched before any
  // second split, so that the short last splits of long pairs come last
  const int kvh = blockIdx.x, seq = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Positions [0, P) are attended by the shared-prefix pass (P = 0: none);
  // this CTA covers part of [P, ctx).
  const int P = a.prefix_tokens;
  // the two tensor maps: fetched while the grid waits for its inputs
  if (warp == 0 && lane < 2)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(lane ? &vmap : &kmap))
                 : "memory");
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: nothing that kernel may write is read before it has completed.
  // Behind the shared-prefix pass, which itself waits for every kernel
  // before it and then lets this grid start on the SMs it leaves free,
  // nothing is waited for: both grids write partials, and the last CTA of
  // this grid to finish waits for the pass, so that the grid never completes
  // before it (the merge kernel after this grid reads the pass's partials).
  if (P == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  // Behind a shared prefix the merge kernel that follows may be scheduled as
  // soon as every CTA of this grid is running: it waits for this grid to
  // complete before it reads anything, and holds only slots this grid no
  // longer needs.
  if (P > 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto finish = [&]() {
    if (P > 0 && threadIdx.x == 0) {
      const int total = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
      if (atomicAdd(a.done, 1) == total - 1) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        atomicExch(a.done, 0);
      }
    }
  };
  const int g = lane >> 2, q4 = lane & 3;
  const int G = a.group;
  const int32_t* trow = a.tables + static_cast<size_t>(seq) * a.max_blocks;
  // Split 0 starts at position P whatever the length, so its query rows and
  // the block ids of its first NS tiles (one per lane of warp 0) are fetched
  // together with the length instead of after it; its first copies then go
  // out without waiting for the rest of the CTA.
  constexpr int kPre = NS * BPT;
  static_assert(kPre <= 32, "one lane per early block id");
  const bool early = split == 0;
  int pre = -1;
  if (early && warp == 0 && lane < kPre && P / T + lane < a.max_blocks) pre = trow[P / T + lane];
  uint32_t qa[KS][HC ? 2 : 4];
  const typename Q::raw* qrows = static_cast<const typename Q::raw*>(a.q) +
      (static_cast<size_t>(seq) * a.num_q_heads + static_cast<size_t>(kvh) * G) * D;
  auto load_query = [&]() {
    if constexpr (HC) load_qt<KV, Q, D>(qa, qrows, G, g, q4);
    else load_q<KV, Q, D>(qa, qrows, G, g, q4);
  };
  if (early) load_query();
  const HeadScales sc = head_scales(a.head_scales, a.num_kv_heads, kvh, a.softmax_scale,
                                    a.qk_scale, a.v_scale, a.k_inv, a.v_inv);
  const int ctx = a.ctx_lens[seq];
  const bool bad_ctx = ctx < 0 || ctx > a.max_blocks * T || (P > 0 && ctx <= P);
  const int own = bad_ctx ? 0 : ctx - P;  // positions this kernel attends
  const int nsplit = bad_ctx ? 1 : max(1, (own + a.partition - 1) / a.partition);
  if (split >= nsplit) {
    finish();
    return;
  }
  const size_t head0 = static_cast<size_t>(seq) * a.num_q_heads + static_cast<size_t>(kvh) * G;
  // The pair's n_t tiles are shared out evenly: split i takes tiles
  // [i n_t / nsplit, (i + 1) n_t / nsplit), at most partition / 64 of them.
  // Near-equal pieces keep the longest units of the grid on pairs that need
  // no merge, and the boundaries still depend only on the length.
  const int64_t n_t = (own + kTile - 1) / kTile;
  const int t_begin = P + static_cast<int>(split * n_t / nsplit) * kTile;
  const int t_end = bad_ctx ? P : min(P + static_cast<int>((split + 1) * n_t / nsplit) * kTile, ctx);
  const int first_blk = t_begin / T;
  const int n_blk = (t_end - t_begin + T - 1) / T;
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;                                            // NS * kStageBytes
  int32_t* s_tab = reinterpret_cast<int32_t*>(smem + NS * G_::kStageBytes);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_tab + kMaxTableEntries);
  __shared__ int s_bad, s_last;  // s_bad: PKV_DEVICE_* bits, written by thread 0 only

  static_assert(NS * G_::kStageBytes >= (2 * kWarps * 16 + kWarps * 16 * D) * 4,
                "the warp merge reuses the stage buffers");
  if (tid == 0) {
    s_bad = bad_ctx ? kBadLength : 0;
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&s_bar[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  // the split's block ids (split 0: those past warp 0's early ones)
  for (int i = (early ? kPre : 0) + tid; i < n_blk; i += kThreads) s_tab[i] = trow[first_blk + i];

  // Fused slot write: the split holding position ctx - 1 stores the step's
  // token of its KV head before any copy is issued (a block never spans two
  // splits, and other heads' rows are disjoint, so no other CTA reads it).
  // Warp 0 writes, and issues every copy after it.
  constexpr int kUnits = D / 8;
  static_assert(2 * kUnits <= 32, "warp 0 writes the step's K and V rows");
  if (a.k_new != nullptr && !bad_ctx && ctx > 0 && split == nsplit - 1 && warp == 0) {
    const int p = ctx - 1;
    const int lb = p / T - first_blk;  // its block within the split
    int blk = __shfl_sync(0xffffffffu, pre, lb & 31);
    if (!(early && lb < kPre)) blk = trow[p / T];
    if (blk >= 0 && blk < a.num_blocks && lane < 2 * kUnits) {
      const int which = lane / kUnits, d0 = (lane % kUnits) * 8;
      const size_t src = (static_cast<size_t>(seq) * a.num_kv_heads + kvh) * D + d0;
      const size_t dst = ((static_cast<size_t>(blk) * a.num_kv_heads + kvh) * T + p % T) * D + d0;
      store8<Q, KV>(static_cast<const typename Q::raw*>(which ? a.v_new : a.k_new) + src,
                    static_cast<typename KV::raw*>(const_cast<void*>(which ? a.v_cache : a.k_cache)) + dst,
                    which ? sc.v_inv : sc.k_inv);
      asm volatile("fence.proxy.async.global;" ::: "memory");  // before the TMA reads it
    }
  }

  // ---------------------------------------------------------- producer
  // Warp 0 refills a stage with one warp instruction: lane l issues box l
  // (block l / 2, K|V), which starts the tile's boxes together instead of one
  // after another from a single thread.
  constexpr int BPB = BPT * 2;  // boxes per tile
  static_assert(BPB <= 32, "one lane per box");
  auto issue = [&](int tile) {
    const int s = tile % NS;
    uint8_t* kt = stages + s * G_::kStageBytes;
    const int lb0 = (tile * kTile) / T;  // first logical block of the tile within the split
    const int blk = lane / 2, isv = lane & 1;
    int phys = -1;
    bool inb = false;
    if (lane < BPB && lb0 + blk < n_blk) {
      inb = true;
      phys = s_tab[lb0 + blk];
    }
    const bool good = inb && phys >= 0 && phys < a.num_blocks;
    const unsigned okmask = __ballot_sync(0xffffffffu, good);
    const unsigned badmask = __ballot_sync(0xffffffffu, inb && !good);
    const uint32_t bar = smem_u32(&s_bar[s]);
    if (lane == 0) {
      if (badmask) s_bad |= kBadTable;
      mbar_arrive_expect_tx(bar, __popc(okmask) * static_cast<uint32_t>(kBoxBytes));
    }
    __syncwarp();
    if (good)
      tma_box<KV, D>(smem_u32(kt + (isv ? G_::kTileBytes : 0) + blk * kBoxBytes), isv ? &vmap : &kmap,
                     (phys * a.num_kv_heads + kvh) * T, bar);
  };
  if (early && warp == 0) {
    // the early block ids: to shared memory (the refills and the table checks
    // read them there), then the first tiles' copies
    if (lane < kPre && lane < n_blk) s_tab[lane] = pre;
    __syncwarp();
    for (int t = 0; t < NS && t < n_tiles; ++t) issue(t);
  }
  if (!early) load_query();
  __syncthreads();
  if (!early && warp == 0)
    for (int t = 0; t < NS && t < n_tiles; ++t) issue(t);

  // ---------------------------------------------------------- consumers
  State st;
  st.reset();
  bool timed_out = false;
  int stalled_at = -1;
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int s = tile % NS;
    const uint32_t parity = (tile / NS) & 1;
    const bool arrived = stage_wait(smem_u32(&s_bar[s]), parity, a.wait_ns);
    const uint8_t* kt = stages + s * G_::kStageBytes;
    uint8_t* vt = stages + s * G_::kStageBytes + G_::kTileBytes;
    const int row0 = warp * 16;
    const int tok0 = t_begin + tile * kTile + row0;
    const int nvalid = min(16, t_end - tok0);
    bool zeroed = false;
    if (arrived && nvalid > 0) {
      if constexpr (HC) zeroed = tile_step_t<KV, D>(st, qa, kt, vt, row0, nvalid, sc.qk, lane);
      else zeroed = tile_step<KV, D>(st, qa, kt, vt, row0, nvalid, sc.qk, lane);
    }
    if (zeroed) fence_proxy_async();  // the zeroed rows, before the slot is refilled by TMA
    if (__syncthreads_or(!arrived)) {
      timed_out = true;
      stalled_at = tile;
      break;
    }
    if (warp == 0 && tile + NS < n_tiles) issue(tile + NS);
  }

  if (timed_out) {
    // wait (bounded) for the copies still in flight, tiles stalled_at ..
    // stalled_at + NS - 1, before the CTA's shared memory can be reused
    if (tid == 0) {
      s_bad |= kTimeout;
      for (int t = stalled_at; t < n_tiles && t < stalled_at + NS; ++t)
        mbar_wait(smem_u32(&s_bar[t % NS]), (t / NS) & 1, kDrainNs);
    }
    __syncthreads();
  }

  // ---------------------------------------------------- merge the warps
  float* mS = reinterpret_cast<float*>(smem);  // stages are idle now
  float* lS = mS + kWarps * 16;
  float* oS = lS + kWarps * 16;                // [warp][16 rows][D]
  if constexpr (HC) publish_t<KV, D>(st, mS, lS, oS, warp, G, 16, lane);
  else publish<KV, D>(st, mS, lS, oS, warp, G, 16, lane);
  __syncthreads();

  const int bad_bits = s_bad;
  if (tid == 0 && bad_bits != 0 && a.status != nullptr) atomicOr(a.status, bad_bits);
  const bool any_bad = bad_bits != 0;
  constexpr int kCap = NS * G_::kStageBytes / 4;  // floats of stage memory
  // A lone split writes the output unless a shared-prefix partial joins it.
  const bool direct = nsplit == 1 && P == 0;
  for (int i = tid; i < G * D; i += kThreads) {
    const int row = i / D, d = i % D;
    float M, L, A;
    combine_warps(mS, lS, oS, kWarps, 16, row, d, D, M, L, A);
    A *= sc.v;
    if (direct) {
      const float out = any_bad ? CUDART_NAN_F : (L > 0.f ? A / L : 0.f);
      store_elem<Q>(a.out, (head0 + row) * D + d, out);
    } else {
      const size_t pidx = (head0 + row) * a.max_splits + split;
      a.ws_acc[pidx * D + d] = any_bad ? CUDART_NAN_F : A;
      if (d == 0) {
        a.ws_m[pidx] = M;
        a.ws_l[pidx] = any_bad ? CUDART_NAN_F : L;
      }
    }
  }

  if (direct) return;
  // behind a shared-prefix pass the merge kernel that follows merges every
  // partial (the units here are short: counting in would cost each CTA the
  // fence and atomic latency at its end)
  if (P > 0) {
    finish();
    return;
  }

  // ------------------------------------------- split-K: the last CTA merges
  // Each CTA counts itself in (an atomic counter, never a wait on another
  // CTA); the last of the pair's splits to arrive combines their partials
  // and resets the counter.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[static_cast<size_t>(seq) * a.num_kv_heads + kvh], 1);
    s_last = prev == nsplit - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_splits<Q, D, kThreads>(a, head0, nsplit, a.max_splits, 0, reinterpret_cast<float*>(smem), kCap);
  if (tid == 0) atomicExch(&a.counters[static_cast<size_t>(seq) * a.num_kv_heads + kvh], 0);
}

template <typename KV, int D, int NS, int W = kWarps>
constexpr int smem_bytes() {
  return NS * Geom<KV, D, W>::kStageBytes + max_table_entries<W>() * 4 + NS * 8 + 1024;
}

}  // namespace tc

// Launch the tensor-core decode kernel for one (cache, q) dtype pair.
template <typename KV, typename Q>
pkv_status launch_decode_tc(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pkv
