// Stream-K decode attention on the tensor cores: the split kernel's tile
// pipeline with the work cut into equal slices.
//
// Same result as the other decode kernels (the katajob Q&A, "The paging
// idea": keys and values gathered through the block table), scheduled so that
// the whole call is one wave of equally loaded CTAs:
//
//  * The work is the list of 64-token tiles of every (sequence, KV head) pair
//    ("pair"), in (sequence, head, tile) order.  The grid is three CTAs per SM
//    (all resident at once); CTA c takes the contiguous slice
//    [c*W/C, (c+1)*W/C) of the W tiles, so every CTA moves the same number of
//    tiles whatever the length mix, and no CTA waits for another.
//  * Inside a CTA the pipeline is the split kernel's: four warps, a 64 KiB
//    ring of 2 (16-bit, head_dim 128) or 4 stages of one tile's K and V,
//    fetched as one TMA box of T rows (all their bytes) per (block, K|V)
//    by the lanes of warp 0, which refills a stage as soon as the four warps
//    have consumed it.  The block ids of the next tile are loaded one tile
//    ahead, so table reads never sit between a free stage and its refill.
//  * The tile counts of all sequences and their prefix sum are formed in the
//    ring before the first copy; afterwards each cursor carries the running
//    tile base of its sequence.
//  * At the end of a pair's tiles in this CTA ("segment") the four warps'
//    states are folded into warp 0 through one warp-sized buffer, in fragment
//    order.  A pair the CTA holds entirely is written out directly; a pair
//    shared with neighbouring CTAs is written as a partial (max, sum,
//    unnormalised output) to the CTA's first or last partial slot (only a
//    slice's first and last pairs can be shared).  After its last tile the
//    CTA counts itself in on each shared pair (an atomic counter, never a
//    wait), and the last of the pair's CTAs to arrive merges the pieces,
//    writes the output and resets the counter; doing this after the loop
//    keeps those global round trips off the copy stream.
//  * Sequences with no tiles (context 0, or an invalid length) get a zero (or
//    NaN) output from CTA (sequence mod C).
//  * Every mbarrier wait is bounded in time; after a stall nothing more is
//    copied or waited for, every remaining segment of the slice is published
//    as NaN (so that the merges of shared pairs still complete), and the CTA
//    waits (bounded) for its copies in flight before it exits.
#pragma once

#include "attention_tc.cuh"

namespace pkv {
namespace tc {

constexpr int kStreamCtasPerSm = 3;
constexpr int kStreamRingBytes = 65536;
constexpr int kCtxWindow = 64;  // context lengths of a slice's first sequences kept in shared memory

template <typename KV, int D>
constexpr int stream_stages() {
  return kStreamRingBytes / Geom<KV, D>::kStageBytes;
}

// One warp's state in fragment order, lane-major: o[D/8][4], m[2], l[2].
template <int D>
constexpr int fold_floats() {
  return (D / 8 * 4 + 4) * 32;
}

template <typename KV, int D>
constexpr int stream_smem_bytes() {
  return 1024 + kStreamRingBytes + fold_floats<D>() * 4 + stream_stages<KV, D>() * 8;
}

struct StreamCursor {
  int s, h, j, nt, base;  // sequence, KV head, tile within the pair, tiles per head, cum tiles before s
};

struct Split {
  int base, rem;
  __device__ __forceinline__ int start(int c) const { return c * base + min(c, rem); }
  __device__ __forceinline__ int owner(int t) const {
    const int big = rem * (base + 1);
    return t < big ? t / (base + 1) : rem + (t - big) / base;
  }
};

template <typename KV, typename Q, int D, int T>
__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm)
    decode_stream_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap) {
  using G_ = Geom<KV, D>;
  constexpr int NS = stream_stages<KV, D>();
  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  constexpr int BPT = kTile / T;                 // blocks per tile
  constexpr int kBoxBytes = T * G_::kRowBytes;    // one (block, head) box: all its slabs
  constexpr int BPB = BPT * 2;                   // boxes per tile
  constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  constexpr unsigned FULL = 0xffffffffu;
  static_assert(NS >= 2 && NS * G_::kStageBytes == kStreamRingBytes, "ring of whole stages");
  static_assert(BPB <= 32, "one lane per box");

  const int C = gridDim.x, c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;
  const int B = a.num_seqs, NKV = a.num_kv_heads, G = a.group, HQ = a.num_q_heads;
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: nothing that kernel may write is read before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int max_ctx = a.max_blocks * T;
  const int PS = G * (D + 2);  // floats of one partial slot

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* fold = reinterpret_cast<float*>(ring + kStreamRingBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(fold + fold_floats<D>());
  __shared__ int s_ctx[kCtxWindow];
  __shared__ int s_wsum[kWarps];
  __shared__ int s_bad[NS];
  __shared__ int s_ids[NS][32];  // block ids of the coming tiles, one per box lane
  __shared__ int s_last[2];

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&full[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  auto tiles_of = [&](int v) { return (v <= 0 || v > max_ctx) ? 0 : (v + kTile - 1) / kTile; };

  // ---- tiles per sequence and their prefix sum, in the ring (idle until the
  // first copy): cum[s] = N_kv * (tiles of the sequences before s)
  int* cum = reinterpret_cast<int*>(ring);
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int run = 0;
    for (int i = b0; i < b1; ++i) {
      run += tiles_of(a.ctx_lens[i]) * NKV;
      cum[1 + i] = run;
    }
    int x = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    int excl = x - run;
    for (int w = 0; w < warp; ++w) excl += s_wsum[w];
    for (int i = b0; i < b1; ++i) cum[1 + i] += excl;
    if (tid == 0) cum[0] = 0;
    __syncthreads();
  }
  const int W = cum[B];

  // ---- sequences with no tiles: zero output (empty context) or NaN (invalid)
  for (int s = c; s < B; s += C) {
    if (cum[s + 1] != cum[s]) continue;
    const float o = a.ctx_lens[s] == 0 ? 0.f : CUDART_NAN_F;
    for (int i = tid; i < HQ * D; i += kThreads)
      store_elem<Q>(a.out, static_cast<size_t>(s) * HQ * D + i, o);
  }

  // ---- this CTA's slice and its first tile
  const Split sp{W / C, W % C};
  const int start = sp.start(c);
  const int len = sp.base + (c < sp.rem ? 1 : 0);
  StreamCursor cur{0, 0, 0, 1, 0};
  if (len > 0) {
    int lo = 0, hi = B;  // cum[lo] <= start < cum[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cum[mid] <= start) lo = mid;
      else hi = mid;
    }
    cur.s = lo;
    cur.base = cum[lo];
    cur.nt = (cum[lo + 1] - cum[lo]) / NKV;
    const int local = start - cum[lo];
    cur.h = local / cur.nt;
    cur.j = local - cur.h * cur.nt;
  }
  const int s0 = cur.s;
  for (int i = tid; i < kCtxWindow; i += kThreads) s_ctx[i] = s0 + i < B ? a.ctx_lens[s0 + i] : 0;
  fence_proxy_async();  // the ring's generic writes, before TMA reuses it
  __syncthreads();
  if (len == 0) return;

  auto ctx_of = [&](int s) { return s - s0 < kCtxWindow ? s_ctx[s - s0] : __ldg(a.ctx_lens + s); };
  auto advance = [&](StreamCursor& r) {
    if (++r.j < r.nt) return;
    r.j = 0;
    if (++r.h < NKV) return;
    r.h = 0;
    r.base += r.nt * NKV;
    do {
      ++r.s;
      r.nt = r.s < B ? tiles_of(ctx_of(r.s)) : 1;
    } while (r.nt == 0);
  };

  // ---------------------------------------------------------- producer side
  // Lane l < BPB of warp 0 fetches box l of a tile: block l / 2, K (even l)
  // or V (odd l), each box all slabs of the block's T rows of one head.  The block ids of tile t
  // come from s_ids[t % NS], filled by an asynchronous copy (cp.async) issued
  // when tile t - NS was issued, a whole ring ahead, so a table read never
  // sits between a freed stage and its refill.
  const int bx_blk = lane / 2, bx_v = lane & 1;
  constexpr int kNoBox = -1, kBadBox = -2;
  auto box_lb = [&](const StreamCursor& r) {  // logical block of this lane's box, or -1
    const int lb = r.j * BPT + bx_blk;
    return (lane < BPB && lb * T < ctx_of(r.s)) ? lb : -1;
  };
  auto checked = [&](int id) { return (id >= 0 && id < a.num_blocks) ? id : kBadBox; };
  auto fetch_ids = [&](int slot, const StreamCursor& r, bool any) {
    const int lb = any ? box_lb(r) : -1;
    if (lb >= 0)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&s_ids[slot][lane])),
                   "l"(a.tables + static_cast<size_t>(r.s) * a.max_blocks + lb)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto issue = [&](int t, const StreamCursor& r, int id) {
    const int slot = t % NS;
    const unsigned okmask = __ballot_sync(FULL, id >= 0);
    const unsigned badmask = __ballot_sync(FULL, id == kBadBox);
    const uint32_t bar = smem_u32(&full[slot]);
    if (lane == 0) {
      s_bad[slot] = badmask != 0;
      mbar_arrive_expect_tx(bar, __popc(okmask) * static_cast<uint32_t>(kBoxBytes));
    }
    __syncwarp();
    if (id >= 0)
      tma_box<KV, D>(smem_u32(ring + slot * G_::kStageBytes + (bx_v ? G_::kTileBytes : 0) +
                              bx_blk * kBoxBytes),
                     bx_v ? &vmap : &kmap, (id * NKV + r.h) * T, bar);
  };

  StreamCursor icur = cur;  // warp 0: the next tile to issue
  StreamCursor fcur = cur;  // warp 0: the next tile whose ids are fetched
  int issued = 0;
  if (warp == 0) {
    // the first NS tiles: ids loaded directly (all in flight at once)
    int ids[NS];
    StreamCursor cs[NS];
#pragma unroll
    for (int t = 0; t < NS; ++t) {
      cs[t] = icur;
      const int lb = t < len ? box_lb(icur) : -1;
      ids[t] = lb < 0 ? kNoBox
                      : checked(__ldg(a.tables + static_cast<size_t>(icur.s) * a.max_blocks + lb));
      if (t + 1 < len) advance(icur);
    }
#pragma unroll
    for (int t = 0; t < NS; ++t)
      if (t < len) issue(t, cs[t], ids[t]);
    issued = min(NS, len);
    // ids of tiles NS .. 2 NS - 1, one copy group per tile
    fcur = icur;
#pragma unroll
    for (int t = NS; t < 2 * NS; ++t) {
      fetch_ids(t % NS, fcur, t < len);
      if (t + 1 < len) advance(fcur);
    }
  }

  // ---------------------------------------------------------- consumers
  WarpState<D> st;
  st.reset();
  uint32_t qa[KS][4];
  auto q_rows = [&](const StreamCursor& r) {
    return static_cast<const typename Q::raw*>(a.q) +
           (static_cast<size_t>(r.s) * HQ + static_cast<size_t>(r.h) * G) * D;
  };
  load_q<KV, Q, D>(qa, q_rows(cur), G, g, q4);
  auto scales_of = [&](const StreamCursor& r) {
    return head_scales(a.head_scales, a.num_kv_heads, r.h, a.softmax_scale, a.qk_scale, a.v_scale,
                       a.k_inv, a.v_inv);
  };
  HeadScales sc = scales_of(cur);
  bool aborted = false, seg_bad = false, first_seg = true;
  int stalled_at = len, seg_j0 = cur.j;
  StreamCursor shared_pairs[2];  // a slice shares at most its first and its last pair
  int n_shared = 0;

  for (int k = 0; k < len; ++k) {
    const int slot = k % NS;
    const bool arrived = !aborted && mbar_wait(smem_u32(&full[slot]), (k / NS) & 1, kWaitNs);
    const int nvalid = min(16, ctx_of(cur.s) - (cur.j * kTile + warp * 16));
    uint8_t* kt = ring + slot * G_::kStageBytes;
    uint8_t* vt = kt + G_::kTileBytes;
    if (arrived && nvalid > 0 &&
        tile_step<KV, D>(st, qa, kt, vt, warp * 16, nvalid, sc.qk, lane))
      fence_proxy_async();  // the zeroed rows, before the slot is refilled by TMA
    seg_bad |= !arrived || s_bad[slot] != 0;
    if (__syncthreads_or(!arrived) && !aborted) {
      aborted = true;
      stalled_at = k;
    }
    if (warp == 0 && !aborted && issued < len) {
      // the copy group of this tile's ids is followed by NS - 1 newer ones
      asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");
      const int t = issued;
      const int lb = box_lb(icur);
      issue(t, icur, lb < 0 ? kNoBox : checked(s_ids[t % NS][lane]));
      fetch_ids(t % NS, fcur, t + NS < len);
      if (t + NS + 1 < len) advance(fcur);
      if (++issued < len) advance(icur);
    }

    if (cur.j == cur.nt - 1 || k == len - 1) {
      // ------------------------------------------------ end of a segment
      const bool complete = seg_j0 == 0 && cur.j == cur.nt - 1;
      // fold warps 3, 2, 1 into warp 0: M = max, f = 2^(m - M), l and o rescaled
#pragma unroll 1
      for (int w = kWarps - 1; w >= 1; --w) {
        if (warp == w) {
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) fold[(n * 4 + e) * 32 + lane] = st.o[n][e];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            fold[(NT * 4 + h) * 32 + lane] = st.m[h];
            fold[(NT * 4 + 2 + h) * 32 + lane] = st.l[h];
          }
        }
        __syncthreads();
        if (warp == 0) {
          float fa[2], fb[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float mo = fold[(NT * 4 + h) * 32 + lane];
            const float lo = fold[(NT * 4 + 2 + h) * 32 + lane];
            const float M = fmaxf(st.m[h], mo);
            fa[h] = st.m[h] == -CUDART_INF_F ? 0.f : exp2f(st.m[h] - M);
            fb[h] = mo == -CUDART_INF_F ? 0.f : exp2f(mo - M);
            st.l[h] = st.l[h] * fa[h] + lo * fb[h];
            st.m[h] = M;
          }
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              st.o[n][e] = st.o[n][e] * fa[e >> 1] + fold[(n * 4 + e) * 32 + lane] * fb[e >> 1];
        }
        __syncthreads();
      }

      const size_t head0 = static_cast<size_t>(cur.s) * HQ + static_cast<size_t>(cur.h) * G;
      if (warp == 0) {
        float* part = a.ws_part + static_cast<size_t>(2 * c + (first_seg ? 0 : 1)) * PS;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float L = st.l[h];
          L += __shfl_xor_sync(FULL, L, 1);
          L += __shfl_xor_sync(FULL, L, 2);
          const int row = g + 8 * h;
          if (row >= G) continue;
          if (complete) {
            const float inv = (L > 0.f || L != L) ? sc.v / L : 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
              for (int jj = 0; jj < 2; ++jj)
                store_elem<Q>(a.out, (head0 + row) * D + out_col<kFp8>(n, jj, q4),
                              seg_bad ? CUDART_NAN_F : st.o[n][2 * h + jj] * inv);
          } else {
            float* pr = part + row * (D + 2);
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
              for (int jj = 0; jj < 2; ++jj)
                pr[2 + out_col<kFp8>(n, jj, q4)] =
                    seg_bad ? CUDART_NAN_F : st.o[n][2 * h + jj] * sc.v;
            if (q4 == 0) {
              pr[0] = st.m[h];
              pr[1] = seg_bad ? CUDART_NAN_F : L;
            }
          }
        }
      }
      // a shared pair is merged after the loop, when the ring is idle: its
      // fence, counter and merge are global round trips that would otherwise
      // stop this CTA's stream for several microseconds under full load
      if (!complete && n_shared < 2) shared_pairs[n_shared++] = cur;
      st.reset();
      seg_bad = false;
      first_seg = false;
      if (k + 1 < len) {
        advance(cur);
        seg_j0 = cur.j;
        load_q<KV, Q, D>(qa, q_rows(cur), G, g, q4);
        sc = scales_of(cur);
      }
    } else {
      advance(cur);
    }
  }

  // ---- after a stall: wait (bounded) for the copies still in flight (the
  // ring is reused below)
  if (aborted && tid == 0)
    for (int t = stalled_at; t < issued; ++t)
      mbar_wait(smem_u32(&full[t % NS]), (t / NS) & 1, kDrainNs);
  if (warp == 0) asm volatile("cp.async.wait_all;" ::: "memory");

  // ---- pairs shared with neighbouring CTAs: the last CTA to arrive merges
  // the pieces (max, sum and unnormalised output of each CTA's part) and
  // resets the pair's counter.  Partial slot 0 of a CTA holds its first
  // segment, slot 1 its last.  Every step here is a global round trip, so
  // the CTA counts itself in on both pairs at once and gathers all pieces of
  // a pair with independent loads before combining them.
  if (n_shared == 0) return;
  __threadfence();  // this thread's partial stores, before the counters
  __syncthreads();
  if (lane == 0 && warp < n_shared) {
    const StreamCursor& pr = shared_pairs[warp];
    const int P0 = pr.base + pr.h * pr.nt;
    const int c0 = sp.owner(P0), c1 = sp.owner(P0 + pr.nt - 1);
    s_last[warp] = atomicAdd(a.counters + static_cast<size_t>(pr.s) * NKV + pr.h, 1) == c1 - c0;
  }
  __syncthreads();
  for (int r = 0; r < n_shared; ++r) {
    if (!s_last[r]) continue;
    __threadfence();
    const StreamCursor pr = shared_pairs[r];
    const int P0 = pr.base + pr.h * pr.nt;
    const int c0 = sp.owner(P0), c1 = sp.owner(P0 + pr.nt - 1);
    const size_t out0 = (static_cast<size_t>(pr.s) * HQ + static_cast<size_t>(pr.h) * G) * D;
    // piece ci (CTA c0 + ci) is CTA c0's last segment unless its slice starts at P0
    auto piece = [&](int ci) {
      const int cc = c0 + ci;
      const int which = (ci == 0 && sp.start(cc) != P0) ? 1 : 0;
      return a.ws_part + static_cast<size_t>(2 * cc + which) * PS;
    };
    const int nc = c1 - c0 + 1;
    const int total = nc * PS;  // even: PS = G * (D + 2)
    if (total <= kStreamRingBytes / 4) {
      float* stage = reinterpret_cast<float*>(ring);
      constexpr int kU = 16;  // float2 loads in flight per thread
      for (int i0 = 0; i0 < total / 2; i0 += kU * kThreads) {
        float2 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = i0 + u * kThreads + tid;
          if (i < total / 2) {
            const int ci = (2 * i) / PS, off = 2 * i - ci * PS;
            v[u] = __ldcg(reinterpret_cast<const float2*>(piece(ci) + off));
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = i0 + u * kThreads + tid;
          if (i < total / 2) reinterpret_cast<float2*>(stage)[i] = v[u];
        }
      }
      __syncthreads();
      for (int e = tid; e < G * D; e += kThreads) {
        const int row = e / D, d = e - row * D;
        float M = -CUDART_INF_F;
        for (int ci = 0; ci < nc; ++ci) M = fmaxf(M, stage[ci * PS + row * (D + 2)]);
        float L = 0.f, A = 0.f;
        if (M != -CUDART_INF_F) {
          for (int ci = 0; ci < nc; ++ci) {
            const float* pp = stage + ci * PS + row * (D + 2);
            const float f = exp2f(pp[0] - M);
            L = fmaf(pp[1], f, L);
            A = fmaf(pp[2 + d], f, A);
          }
        }
        store_elem<Q>(a.out, out0 + e, (L > 0.f || L != L) ? A / L : 0.f);
      }
    } else {
      // very long pairs (pieces larger than the ring): combine from L2 directly
      for (int e = tid; e < G * D; e += kThreads) {
        const int row = e / D, d = e - row * D;
        float M = -CUDART_INF_F;
        for (int ci = 0; ci < nc; ++ci) M = fmaxf(M, __ldcg(piece(ci) + row * (D + 2)));
        float L = 0.f, A = 0.f;
        if (M != -CUDART_INF_F) {
          for (int ci = 0; ci < nc; ++ci) {
            const float* pp = piece(ci) + row * (D + 2);
            const float f = exp2f(__ldcg(pp) - M);
            L = fmaf(__ldcg(pp + 1), f, L);
            A = fmaf(__ldcg(pp + 2 + d), f, A);
          }
        }
        store_elem<Q>(a.out, out0 + e, (L > 0.f || L != L) ? A / L : 0.f);
      }
    }
    if (tid == 0) atomicExch(a.counters + static_cast<size_t>(pr.s) * NKV + pr.h, 0);
    __syncthreads();  // the staging area is reused by the next pair
  }
}

}  // namespace tc

// Launch the stream-K tensor-core decode kernel for one (cache, q) dtype pair.
template <typename KV, typename Q>
pkv_status launch_decode_stream(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pkv
