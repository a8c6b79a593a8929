// Prefill (multi-query, causal) attention through block tables on tensor
// cores, and its C entry point.
//
// What it computes (the katajob Q&A, "What the KV cache is": every earlier
// token's key and value serve the attention of the next one; "The paging
// idea": a sequence starts with the blocks of its prompt; "PagedAttention,
// clearly explained": later tokens attend over the cached prompt): the chunk
// of sequence s is its last n_s logical positions, already written to the
// pool; the query at position p attends to positions 0 .. p, keys and values
// gathered through the block table.  A one-token chunk is decode attention.
//
// How, on GB300 (FlashAttention-2 tiling over the paged pool):
//  * One CTA (4 warps) per (64-query tile, query head, sequence); the grid
//    column index counts tiles from the END of the chunk, so the tiles with
//    the most keys are dispatched first.
//  * K/V of 64-token tiles of the head's KV head are fetched as 2-D TMA boxes
//    of T rows x 128 bytes per (block, slab, K|V) into a ring of stages, one
//    lane of warp 0 per box, completion by expect-tx mbarriers; block ids
//    are loaded one tile ahead.  A tile keeps its 128-byte slabs apart, so
//    the 8 rows an ldmatrix reads sit on 8 distinct swizzle phases (with
//    whole 256-byte rows back to back, rows r and r + 4 would share one and
//    every K and V fragment load would take two bank passes; the tile is
//    read 64 times, so that matters here, unlike in decode).
//  * Each warp owns 16 query rows and sweeps all 64 keys of every tile:
//    S = Q K^T by mma.sync m16n8k16 (8 key n-tiles), positions after the
//    row's query masked to -inf, online softmax in the log2 domain on the
//    fragments, O += P V by a second MMA with P reused from registers.  Rows
//    never need a cross-warp merge.  Tiles entirely after a warp's last query
//    are skipped by that warp.
//  * V rows at positions >= ctx (the tail of the last block) are zeroed in
//    shared memory before the P V product (0 * NaN would poison it).
//  * Every mbarrier wait is bounded; a timeout turns the CTA's rows into NaN
//    after waiting (bounded) for the copies in flight.
#include <atomic>
#include <type_traits>

#include "attention.h"
#include "attention_tc.cuh"

namespace pkv {
namespace tc {
namespace {

constexpr int kSlabBytes = kTile * 128;   // one 128-byte column slab of a tile

// Byte offset of 16-byte chunk c of tile row r: slab c / 8, then the row's
// 128-byte line, the chunk index XORed with the row index mod 8 (the
// 128-byte swizzle of a box of 128-byte rows; the tile base is 1024-byte
// aligned).
__device__ __forceinline__ uint32_t swz_slab(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * kSlabBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

}  // namespace


template <typename KV, typename Q, int D, int T, int NS>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using G_ = Geom<KV, D>;
  using raw = typename Q::raw;                  // q and out
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  constexpr bool kBf = std::is_same<KV, BF16>::value;   // MMA type: bf16, else f16
  constexpr bool kOutBf = std::is_same<Q, BF16>::value;
  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  constexpr int BPT = kTile / T;
  constexpr int kBoxBytes = T * 128;              // one (block, slab) box
  constexpr int BPB = BPT * G_::kSlabs * 2;      // boxes per tile
  constexpr unsigned FULL = 0xffffffffu;
  static_assert(BPB <= 32, "one lane per box");

  // Launched as a programmatic dependent of the previous kernel in the
  // stream: nothing that kernel may write is read before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int qt_rev = blockIdx.x, j = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3, li = lane & 7, mi = lane >> 3;
  const int HQ = a.num_q_heads;
  const int ctx = a.ctx_lens[s];
  const int q0 = a.query_start[s];
  const int n = a.query_start[s + 1] - q0;
  if (q0 < 0 || n <= 0 || q0 + n > a.total_q) return;  // no rows this CTA may write
  const bool bad = ctx < 0 || ctx > a.max_blocks * T || n > ctx ||
                   (n + kTile - 1) / kTile > a.max_q_tiles;
  if (bad) {  // invalid lengths: the chunk's rows of head j become NaN
    if (tid == 0 && a.status != nullptr) atomicOr(a.status, kBadLength);
    if (qt_rev == 0)
      for (int i = tid; i < n * D; i += kThreads)
        store_elem<Q>(a.out, (static_cast<size_t>(q0 + i / D) * HQ + j) * D + i % D,
                      CUDART_NAN_F);
    return;
  }
  const int ntq = (n + kTile - 1) / kTile;
  if (qt_rev >= ntq) return;
  const int qt = ntq - 1 - qt_rev;
  const int first = ctx - n;                   // position of the chunk's first query
  const int r_begin = qt * kTile;              // chunk row of the tile's first query
  const int r_end = min(r_begin + kTile, n);
  const int kv_end = first + r_end;            // keys 0 .. kv_end - 1
  const int n_kv_tiles = (kv_end + kTile - 1) / kTile;
  const int kvh = j / a.group;
  const HeadScales hs = head_scales(a.head_scales, a.num_kv_heads, kvh, a.softmax_scale, a.qk_scale,
                                    a.v_scale, 1.f, 1.f);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(ring + NS * G_::kStageBytes);
  __shared__ int s_bad;  // PKV_DEVICE_* bits, written by thread 0 only
  if (tid == 0) {
    s_bad = 0;
    for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&s_bar[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---------------------------------------------------------- producer
  const int bx_blk = lane / (G_::kSlabs * 2), bx_sl = (lane / 2) % G_::kSlabs, bx_v = lane & 1;
  constexpr int kNoBox = -1, kBadBox = -2;
  auto box_id = [&](int t) {
    const int lb = t * BPT + bx_blk;
    if (lane >= BPB || lb * T >= ctx) return kNoBox;
    const int id = __ldg(a.tables + static_cast<size_t>(s) * a.max_blocks + lb);
    return (id >= 0 && id < a.num_blocks) ? id : kBadBox;
  };
  auto issue = [&](int t, int id) {
    const int slot = t % NS;
    const unsigned okmask = __ballot_sync(FULL, id >= 0);
    const unsigned badmask = __ballot_sync(FULL, id == kBadBox);
    const uint32_t bar = smem_u32(&s_bar[slot]);
    if (lane == 0) {
      if (badmask) s_bad |= kBadTable;
      mbar_arrive_expect_tx(bar, __popc(okmask) * static_cast<uint32_t>(kBoxBytes));
    }
    __syncwarp();
    if (id >= 0)
      tma_load_2d(smem_u32(ring + slot * G_::kStageBytes + (bx_v ? G_::kTileBytes : 0) +
                           bx_sl * kSlabBytes + bx_blk * kBoxBytes),
                  bx_v ? &vmap : &kmap, bx_sl * 128, (id * a.num_kv_heads + kvh) * T, bar);
  };
  int nid = kNoBox;
  if (warp == 0) {
    int ids[NS];
#pragma unroll
    for (int t = 0; t < NS; ++t) ids[t] = t < n_kv_tiles ? box_id(t) : kNoBox;
#pragma unroll
    for (int t = 0; t < NS; ++t)
      if (t < n_kv_tiles) issue(t, ids[t]);
    if (NS < n_kv_tiles) nid = box_id(NS);
  }

  // ---------------------------------------------------------- consumers
  // this warp's rows g and g + 8 of 16: chunk rows r_begin + 16 warp + ..
  const int wr0 = r_begin + warp * 16;
  const bool warp_any = wr0 < r_end;
  int qpos[2];
  bool rvalid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = wr0 + g + 8 * h;
    rvalid[h] = r < r_end;
    qpos[h] = first + (rvalid[h] ? r : r_begin);  // an invalid row behaves like the tile's first
  }
  const int warp_last = first + min(wr0 + 15, r_end - 1);
  uint32_t qa[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo = 0, hi = 0;
      if (rvalid[h]) {
        const raw* qrow =
            static_cast<const raw*>(a.q) + (static_cast<size_t>(q0 + wr0 + g + 8 * h) * HQ + j) * D;
        if constexpr (!kFp8) {
          const uint32_t* qp = reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * q4);
          lo = qp[0];
          hi = qp[4];
        } else {
          // f16, head_dim permuted within the 16-element step so that one
          // 4-byte K load serves both halves of the k-step
          float f[4];
          LoadF32<Q, 4>::run(qrow + 16 * ks + 4 * q4, f);
          lo = pack2<false>(f[0], f[1]);
          hi = pack2<false>(f[2], f[3]);
        }
      }
      qa[ks][h] = lo;
      qa[ks][2 + h] = hi;
    }

  float o[NT][4];
#pragma unroll
  for (int c = 0; c < NT; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;
  float m[2] = {-CUDART_INF_F, -CUDART_INF_F}, l[2] = {0.f, 0.f};

  bool timed_out = false;
  int stalled_at = -1;
  for (int t = 0; t < n_kv_tiles; ++t) {
    const int slot = t % NS;
    const bool arrived = mbar_wait(smem_u32(&s_bar[slot]), (t / NS) & 1, kWaitNs);
    uint8_t* kt = ring + slot * G_::kStageBytes;
    uint8_t* vt = kt + G_::kTileBytes;
    const int tile_base = t * kTile;
    if (tile_base + kTile > ctx) {
      // zero V rows at positions >= ctx (never written, or another block's)
      const int z0 = ctx - tile_base;
      const int nz = (kTile - z0) * G_::kSlabs * 8;
      for (int i = tid; i < nz; i += kThreads) {
        const int r = z0 + i / (G_::kSlabs * 8), c = i % (G_::kSlabs * 8);
        *reinterpret_cast<uint4*>(vt + swz_slab(r, c)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();  // before the slot is refilled by TMA
      __syncthreads();
    }
    if (arrived && warp_any && tile_base <= warp_last) {
      const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
      // S = Q K^T: 8 n-tiles of 8 keys
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        const int r = 8 * nt + li;
        if constexpr (!kFp8) {
#pragma unroll
          for (int ks = 0; ks < KS; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + swz_slab(r, 2 * ks + mi), b0, b1, b2, b3);
            mma16816<kBf>(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma16816<kBf>(sc[nt], qa[ks + 1][0], qa[ks + 1][1], qa[ks + 1][2], qa[ks + 1][3], b2, b3);
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < KS; c0 += 4) {
            uint32_t w[4];
            ldsm_x4(kbase + swz_slab(r, c0 + mi), w[0], w[1], w[2], w[3]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int ks = c0 + jj;
              mma16816<false>(sc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3],
                              e4m3x2_f16x2(w[jj] & 0xffffu), e4m3x2_f16x2(w[jj] >> 16));
            }
          }
        }
      }
      // causal mask and online softmax, rows g (h = 0) and g + 8 (h = 1)
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int pos = tile_base + 8 * nt + 2 * q4 + jj;
            float v = sc[nt][2 * h + jj] * hs.qk;
            v = pos <= qpos[h] ? v : -CUDART_INF_F;
            sc[nt][2 * h + jj] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
        const float mn = fmaxf(m[h], mx);
        corr[h] = exp2f(m[h] - mn);
        m[h] = mn;
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const float e = exp2f(sc[nt][2 * h + jj] - mn);
            sc[nt][2 * h + jj] = e;
            sum += e;
          }
        l[h] = l[h] * corr[h] + sum;
      }
#pragma unroll
      for (int c = 0; c < NT; ++c) {
        o[c][0] *= corr[0];
        o[c][1] *= corr[0];
        o[c][2] *= corr[1];
        o[c][3] *= corr[1];
      }
      // O += P V: 4 k-steps of 16 keys
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t pa0 = pack2<kBf>(sc[2 * kk][0], sc[2 * kk][1]);
        const uint32_t pa1 = pack2<kBf>(sc[2 * kk][2], sc[2 * kk][3]);
        const uint32_t pa2 = pack2<kBf>(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        const uint32_t pa3 = pack2<kBf>(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const int rv = 16 * kk + (mi & 1) * 8 + li;
        if constexpr (!kFp8) {
#pragma unroll
          for (int c = 0; c < NT; c += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vbase + swz_slab(rv, c + (mi >> 1)), b0, b1, b2, b3);
            mma16816<kBf>(o[c], pa0, pa1, pa2, pa3, b0, b1);
            mma16816<kBf>(o[c + 1], pa0, pa1, pa2, pa3, b2, b3);
          }
        } else {
#pragma unroll
          for (int c = 0; c < D / 16; c += 2) {
            uint32_t w0, w1, w2, w3;  // (keys 0-7, chunk c), (8-15, c), (0-7, c + 1), (8-15, c + 1)
            ldsm_x4_t(vbase + swz_slab(rv, c + (mi >> 1)), w0, w1, w2, w3);
            const uint32_t x0 = prmt(w0, 0x3120), x1 = prmt(w1, 0x3120);
            const uint32_t x2 = prmt(w2, 0x3120), x3 = prmt(w3, 0x3120);
            // chunk c: even head_dim index -> n-tile 2c, odd -> 2c + 1
            mma16816<false>(o[2 * c], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x0 & 0xffffu),
                            e4m3x2_f16x2(x1 & 0xffffu));
            mma16816<false>(o[2 * c + 1], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x0 >> 16),
                            e4m3x2_f16x2(x1 >> 16));
            mma16816<false>(o[2 * c + 2], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x2 & 0xffffu),
                            e4m3x2_f16x2(x3 & 0xffffu));
            mma16816<false>(o[2 * c + 3], pa0, pa1, pa2, pa3, e4m3x2_f16x2(x2 >> 16),
                            e4m3x2_f16x2(x3 >> 16));
          }
        }
      }
    }
    if (__syncthreads_or(!arrived)) {
      timed_out = true;
      stalled_at = t;
      break;
    }
    if (warp == 0 && t + NS < n_kv_tiles) {
      issue(t + NS, nid);
      if (t + NS + 1 < n_kv_tiles) nid = box_id(t + NS + 1);
    }
  }

  if (timed_out && tid == 0) {
    // wait (bounded) for the copies still in flight before the CTA exits
    s_bad |= kTimeout;
    for (int t = stalled_at; t < n_kv_tiles && t < stalled_at + NS; ++t)
      mbar_wait(smem_u32(&s_bar[t % NS]), (t / NS) & 1, kDrainNs);
  }
  __syncthreads();
  const bool any_bad = s_bad != 0;
  if (tid == 0 && any_bad && a.status != nullptr) atomicOr(a.status, s_bad);

  // ---------------------------------------------------------- epilogue
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float L = l[h];
    L += __shfl_xor_sync(FULL, L, 1);
    L += __shfl_xor_sync(FULL, L, 2);
    if (!warp_any || !rvalid[h]) continue;
    const float inv = (L > 0.f || L != L) ? hs.v / L : 0.f;
    raw* orow = static_cast<raw*>(a.out) +
                (static_cast<size_t>(q0 + wr0 + g + 8 * h) * HQ + j) * D;
    if constexpr (!kFp8) {
#pragma unroll
      for (int c = 0; c < NT; ++c) {
        const float x0 = any_bad ? CUDART_NAN_F : o[c][2 * h] * inv;
        const float x1 = any_bad ? CUDART_NAN_F : o[c][2 * h + 1] * inv;
        *reinterpret_cast<uint32_t*>(orow + 8 * c + 2 * q4) = pack2<kOutBf>(x0, x1);
      }
    } else {
      // n-tile n holds head_dim 16 (n / 2) + 4 q4 + 2 jj + (n % 2): the two
      // n-tiles of a pair give adjacent columns
#pragma unroll
      for (int c = 0; c < NT; c += 2)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float x0 = any_bad ? CUDART_NAN_F : o[c][2 * h + jj] * inv;
          const float x1 = any_bad ? CUDART_NAN_F : o[c + 1][2 * h + jj] * inv;
          *reinterpret_cast<uint32_t*>(orow + 16 * (c / 2) + 4 * q4 + 2 * jj) = pack2<kOutBf>(x0, x1);
        }
    }
  }
}

template <typename KV, int D, int NS>
constexpr int prefill_smem_bytes() {
  return 1024 + NS * Geom<KV, D>::kStageBytes + NS * 8;
}

template <typename KV, typename Q, int D, int T>
pkv_status launch_prefill_dt(const PrefillArgs& a, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t st) {
  constexpr int NS = Geom<KV, D>::kStageBytes >= 32768 ? 2 : 4;  // 64 KiB ring
  constexpr int smem = prefill_smem_bytes<KV, D, NS>();
  auto kernel = prefill_tc_kernel<KV, Q, D, T, NS>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: cudaGetDevice", e);
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: cudaFuncSetAttribute", e);
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.max_q_tiles, a.num_q_heads, a.num_seqs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, kmap, vmap);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: launch", e);
  return check_launch("pkv_attention_prefill");
}

}  // namespace tc
}  // namespace pkv

#include "attention_prefill_umma.cuh"

namespace pkv {
namespace tc {

// Process-wide prefill kernel choice (pkv_set_prefill_kernel).
std::atomic<int> g_prefill_choice{PKV_PREFILL_AUTO};

template <typename KV, typename Q, int T>
pkv_status launch_prefill_umma(PrefillArgs a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               int32_t max_query_len, cudaStream_t st) {
  constexpr int smem = umma::smem_bytes<KV>();
  auto kernel = umma::prefill_umma_kernel<KV, Q, T>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: cudaGetDevice", e);
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: cudaFuncSetAttribute", e);
    configured.fetch_or(bit);
  }
  a.max_q_tiles = ((max_query_len + umma::kRows - 1) / umma::kRows + 1) / 2;  // pairs of query tiles
  // up to 256 (sequence, pair) units: ranked longest first in the kernel
  const bool ranked = static_cast<int64_t>(a.num_seqs) * a.max_q_tiles <= umma::kMaxRanked;
  a.ranked = ranked ? 1 : 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = ranked ? dim3(a.num_q_heads, a.num_seqs * a.max_q_tiles, 1)
                       : dim3(a.max_q_tiles, a.num_q_heads, a.num_seqs);
  cfg.blockDim = dim3(umma::threads<KV>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, kmap, vmap);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_prefill: launch", e);
  return check_launch("pkv_attention_prefill (tcgen05)");
}

template <typename KV, typename Q>
pkv_status launch_prefill(const PrefillArgs& a, int D, int T, const CUtensorMap& kmap,
                          const CUtensorMap& vmap, cudaStream_t st) {
  if (D == 128 && T == 16) return launch_prefill_dt<KV, Q, 128, 16>(a, kmap, vmap, st);
  if (D == 128 && T == 32) return launch_prefill_dt<KV, Q, 128, 32>(a, kmap, vmap, st);
  if constexpr (!std::is_same<KV, E4M3>::value) {
    if (D == 64 && T == 16) return launch_prefill_dt<KV, Q, 64, 16>(a, kmap, vmap, st);
    if (D == 64 && T == 32) return launch_prefill_dt<KV, Q, 64, 32>(a, kmap, vmap, st);
  }
  return fail(PKV_ERR_UNSUPPORTED, "pkv_attention_prefill: head_dim/block_size not compiled");
}

}  // namespace tc
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_attention_prefill(void* out, const void* q, int32_t q_dtype,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, int32_t max_blocks,
                                            const int32_t* context_lens,
                                            const int32_t* query_start, int32_t num_seqs,
                                            int32_t total_q, int32_t max_query_len,
                                            int32_t num_q_heads, const pkv_kv_desc* desc,
                                            float softmax_scale, float k_scale, float v_scale,
                                            void* stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || total_q < 0 || max_query_len < 0 || num_q_heads <= 0 || max_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "negative size or no query heads");
  if (num_seqs == 0 || total_q == 0 || max_query_len == 0) return PKV_OK;
  if (num_seqs > 65535 || num_q_heads > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "more than 65535 sequences or query heads per call");
  if (max_blocks == 0) return fail(PKV_ERR_INVALID_ARG, "max_blocks is 0");
  if (num_q_heads % desc->num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  for (const void* p : {static_cast<const void*>(out), q, k_cache, v_cache})
    if (!aligned(p, 16)) return fail(PKV_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4))
    return fail(PKV_ERR_INVALID_ARG, "tables misaligned");
  if (static_cast<int64_t>(max_blocks) * desc->block_size > (int64_t{1} << 30))
    return fail(PKV_ERR_UNSUPPORTED, "context longer than 2^30 tokens");
  if (static_cast<int64_t>(desc->num_blocks) * desc->num_kv_heads * desc->block_size > INT32_MAX)
    return fail(PKV_ERR_UNSUPPORTED, "pool larger than 2^31 rows");
  if (!(softmax_scale == softmax_scale)) return fail(PKV_ERR_INVALID_ARG, "softmax_scale is NaN");
  const int kv = desc->kv_dtype;
  if (!((kv == PKV_BF16 && q_dtype == PKV_BF16) || (kv == PKV_F16 && q_dtype == PKV_F16) ||
        (kv == PKV_E4M3 && (q_dtype == PKV_F16 || q_dtype == PKV_BF16))))
    return fail(PKV_ERR_UNSUPPORTED,
                "pkv_attention_prefill: 16-bit caches with the same q dtype, or E4M3 with f16/bf16 q");
  const int64_t q_tiles = (static_cast<int64_t>(max_query_len) + 63) / 64;
  if (q_tiles > 65535) return fail(PKV_ERR_UNSUPPORTED, "max_query_len too large");

  PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.tables = block_tables;
  a.ctx_lens = context_lens;
  a.query_start = query_start;
  a.max_blocks = max_blocks;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_q_tiles = static_cast<int32_t>(q_tiles);
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = desc->num_kv_heads;
  a.group = num_q_heads / desc->num_kv_heads;
  a.num_blocks = desc->num_blocks;
  const bool fp8 = kv == PKV_E4M3;
  a.qk_scale = softmax_scale * (fp8 ? k_scale : 1.0f) * 1.4426950408889634f;
  a.v_scale = fp8 ? v_scale : 1.0f;
  a.head_scales = desc->head_scales;
  a.softmax_scale = softmax_scale;

  CUtensorMap kmap, vmap;
  st = pool_map(&kmap, k_cache, desc, false);
  if (st == PKV_OK) st = pool_map(&vmap, v_cache, desc, false);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = desc->head_dim, T = desc->block_size;
  // head_dim 128 with a positive softmax scale runs on tcgen05 (E4M3 caches
  // widened to f16 in shared memory) unless the mma.sync kernel is chosen
  // (the tcgen05 kernel folds the softmax scale into the row maximum)
  const int choice = tc::g_prefill_choice.load();
  if (D == 128 && softmax_scale > 0.f && choice != PKV_PREFILL_MMA_SYNC) {
    if (kv == PKV_BF16)
      return T == 16 ? tc::launch_prefill_umma<BF16, BF16, 16>(a, kmap, vmap, max_query_len, s)
                     : tc::launch_prefill_umma<BF16, BF16, 32>(a, kmap, vmap, max_query_len, s);
    if (kv == PKV_F16)
      return T == 16 ? tc::launch_prefill_umma<F16, F16, 16>(a, kmap, vmap, max_query_len, s)
                     : tc::launch_prefill_umma<F16, F16, 32>(a, kmap, vmap, max_query_len, s);
    if (q_dtype == PKV_BF16)
      return T == 16 ? tc::launch_prefill_umma<E4M3, BF16, 16>(a, kmap, vmap, max_query_len, s)
                     : tc::launch_prefill_umma<E4M3, BF16, 32>(a, kmap, vmap, max_query_len, s);
    return T == 16 ? tc::launch_prefill_umma<E4M3, F16, 16>(a, kmap, vmap, max_query_len, s)
                   : tc::launch_prefill_umma<E4M3, F16, 32>(a, kmap, vmap, max_query_len, s);
  }
  if (choice == PKV_PREFILL_TCGEN05)
    return fail(PKV_ERR_UNSUPPORTED, "the tcgen05 prefill kernel needs head_dim 128 and softmax_scale > 0");
  if (kv == PKV_BF16) return tc::launch_prefill<BF16, BF16>(a, D, T, kmap, vmap, s);
  if (kv == PKV_F16) return tc::launch_prefill<F16, F16>(a, D, T, kmap, vmap, s);
  return q_dtype == PKV_F16 ? tc::launch_prefill<E4M3, F16>(a, D, T, kmap, vmap, s)
                            : tc::launch_prefill<E4M3, BF16>(a, D, T, kmap, vmap, s);
}

extern "C" pkv_status pkv_set_prefill_kernel(int32_t kind) {
  if (kind != PKV_PREFILL_AUTO && kind != PKV_PREFILL_MMA_SYNC && kind != PKV_PREFILL_TCGEN05)
    return fail(PKV_ERR_INVALID_ARG, "unknown prefill kernel kind");
  tc::g_prefill_choice.store(kind);
  return PKV_OK;
}
