// Persistent, warp-specialised, stream-K decode attention (tensor cores).
//
// Same result as the other decode kernels (the katajob Q&A, "The paging
// idea": keys and values gathered through the block table), scheduled for
// GB300 so that every SM streams K/V at full rate from launch to finish:
//
//  * Tiles span KV heads.  One block of the pool holds its N_kv heads' T
//    token rows back to back, so HG consecutive heads of a block are one
//    contiguous run of HG * T rows.  A tile is 64 rows: HG heads of
//    64 / (HG * T) blocks, fetched as one 2-D TMA box per (block, 128-byte
//    slab, K|V).  With block size 16 and four or more KV heads that is one
//    8 KB box per slab instead of four 2 KB boxes: the per-box issue cost of
//    the copy engine, not DRAM, limited the one-head tiles.
//  * One CTA per SM for the whole call.  The work is the list of tiles of
//    every (sequence, head group) pair, in (sequence, group, tile) order; CTA
//    c takes the contiguous slice [c*W/C, (c+1)*W/C) of the W tiles, so every
//    CTA moves the same number of tiles whatever the length mix.
//  * Warp 8 is the producer: it walks its slice, takes the block ids of the
//    coming tiles from the table (read one 32-lane window ahead), and issues
//    a batch of tiles' boxes in one warp instruction (one box per lane) into a
//    ring of `stages` slots, completing each slot's "full" mbarrier by byte
//    count.  The first two tiles of each pair also carry the pair's q rows (a
//    bulk copy).  A slot is refilled as soon as its consumers release it
//    ("empty" mbarrier), so the pipeline never drains at pair boundaries.
//  * Warps 0-7 are consumers in two groups of four; group g takes the tiles
//    with an index of parity g, and warp w of a group takes the tile's rows
//    16w .. 16w + 15, i.e. 16 tokens of one head (MMA q.K^T, online softmax,
//    MMA p.V in tile_step()).  At the end of a pair's tiles in this CTA the
//    warps that hold the same head merge their states in shared memory.  A
//    pair the CTA holds entirely is written out directly; a pair shared with
//    neighbouring CTAs is written as a partial (max, sum, unnormalised output)
//    to one of the CTA's two partial slots, and the last of the pair's CTAs to
//    arrive (an atomic counter, never a wait) merges the pieces, writes the
//    output and resets the counter.
//  * The ring depth is a multiple of the group count, so a slot is always
//    consumed by the same group: parity waits only ever target the next phase
//    of a barrier (with slots alternating between groups a group running
//    ahead could wait two phases ahead and see a false completion).
//  * Sequences with no tiles (context 0, or an invalid length) get a zero (or
//    NaN) output from CTA (sequence mod C).
//  * Every mbarrier wait is bounded in time; a stall stops the producer and
//    the consumers' waits, turns the affected outputs into NaN, and the CTA
//    waits (bounded) for its copies in flight before it exits.
#pragma once

#include <climits>

#include "attention_tc.cuh"

namespace pkv {
namespace tc {

constexpr int kGroups = 2;                               // consumer groups
constexpr int kConsumerWarps = kGroups * kWarps;         // 8
constexpr int kProducerWarp = kConsumerWarps;            // warp 8
constexpr int kPersistThreads = (kConsumerWarps + 1) * 32;
constexpr int kPersistMaxStages = 8;

// Bytes of one ring slot's q rows (qrows = HG * G rows of D 16-bit values).
__host__ __device__ constexpr int q_slot_bytes(int qrows, int D) {
  return (qrows * D * 2 + 127) / 128 * 128;
}

// Dynamic shared memory of the persistent kernel (bytes, with alignment slack).
__host__ __device__ constexpr size_t persist_smem_bytes(int stage_bytes, int D, int stages,
                                                        int num_seqs, int group, int qrows) {
  return 1024 + static_cast<size_t>(stages) * (stage_bytes + q_slot_bytes(qrows, D)) +
         (2 * kConsumerWarps * 16 + kConsumerWarps * group * D) * 4 + (2 * num_seqs + 1) * 4 +
         stages * 4 + 8 + 2 * stages * 8;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Named barrier over the consumer warps only (the producer never joins it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

struct Cursor {
  int s, h, j, nt;  // sequence, head group, tile within the pair, tiles of the pair
};

// Tile t of the global list: cum[s] <= t < cum[s + 1] (cum holds groups * tiles).
__device__ __forceinline__ Cursor locate(const int* cum, int B, int ngroups, int t) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= t) lo = mid;
    else hi = mid;
  }
  Cursor r;
  r.s = lo;
  r.nt = (cum[lo + 1] - cum[lo]) / ngroups;
  const int local = t - cum[lo];
  r.h = local / r.nt;
  r.j = local - r.h * r.nt;
  return r;
}

__device__ __forceinline__ void advance(Cursor& r, const int* cum, int ngroups) {
  if (++r.j < r.nt) return;
  r.j = 0;
  if (++r.h < ngroups) return;
  r.h = 0;
  do {
    ++r.s;
  } while (cum[r.s + 1] == cum[r.s]);
  r.nt = (cum[r.s + 1] - cum[r.s]) / ngroups;
}

struct Split {
  int base, rem;
  __device__ __forceinline__ int start(int c) const { return c * base + min(c, rem); }
  __device__ __forceinline__ int owner(int t) const {
    const int big = rem * (base + 1);
    return t < big ? t / (base + 1) : rem + (t - big) / base;
  }
};

template <typename KV, typename Q, int D, int T>
__global__ void __launch_bounds__(kPersistThreads, 1)
    decode_persist_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap) {
  using G_ = Geom<KV, D>;
  constexpr int KS = D / 16;
  constexpr unsigned FULL = 0xffffffffu;

  const int NS = a.stages;
  const int C = gridDim.x, c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.num_seqs, NKV = a.num_kv_heads, G = a.group;
  const int HG = a.hg;                   // KV heads per tile
  const int NHG = NKV / HG;              // head groups
  const int BPT = kTile / (HG * T);      // blocks per tile
  const int TOKS = BPT * T;              // tokens of one head per tile (64 / HG)
  const int box_rows = HG * T;
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * 128u;
  const int QROWS = HG * G;              // q rows of a pair
  const int QB = q_slot_bytes(QROWS, D);
  const int PS = QROWS * (D + 2);        // floats of one partial slot

  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qbuf = ring + static_cast<size_t>(NS) * G_::kStageBytes;
  float* mS = reinterpret_cast<float*>(qbuf + static_cast<size_t>(NS) * QB);
  float* lS = mS + kConsumerWarps * 16;
  float* oS = lS + kConsumerWarps * 16;                            // [warp][G][D]
  int* cum = reinterpret_cast<int*>(oS + kConsumerWarps * G * D);  // B + 1
  int* ctxs = cum + B + 1;                                         // B
  int* sbad = ctxs + B;                                            // NS
  uint64_t* full = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sbad + NS) + 7) &
                                               ~uintptr_t(7));
  uint64_t* empty = full + NS;
  __shared__ int s_wsum[kPersistThreads / 32];
  __shared__ volatile int s_abort;
  __shared__ int s_last, s_segbad;

  // ---- tiles per sequence and their prefix sum (cum[s] = groups * tiles before s)
  const int max_ctx = a.max_blocks * T;
  for (int s = tid; s < B; s += kPersistThreads) {
    const int v = a.ctx_lens[s];
    ctxs[s] = v;
    const int nt = (v <= 0 || v > max_ctx) ? 0 : (v + TOKS - 1) / TOKS;
    cum[s + 1] = nt * NHG;
  }
  if (tid == 0) {
    cum[0] = 0;
    s_abort = 0;
    s_segbad = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kWarps);  // the owning group's four warps
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  __syncthreads();
  {
    const int per = (B + kPersistThreads - 1) / kPersistThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int run = 0;
    for (int i = b0; i < b1; ++i) {
      run += cum[1 + i];
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
    __syncthreads();
  }
  const int W = cum[B];

  // ---- sequences with no tiles: zero output (empty context) or NaN (invalid)
  for (int s = c; s < B; s += C) {
    if (cum[s + 1] != cum[s]) continue;
    const float o = ctxs[s] == 0 ? 0.f : CUDART_NAN_F;
    for (int i = tid; i < a.num_q_heads * D; i += kPersistThreads)
      store_elem<Q>(a.out, static_cast<size_t>(s) * a.num_q_heads * D + i, o);
  }

  const Split sp{W / C, W % C};
  const int start = sp.start(c);
  const int len = sp.base + (c < sp.rem ? 1 : 0);
  if (len == 0) return;
  if (NS < 2 || NS % kGroups != 0) s_abort = 1;  // launch invariant; never true in practice

  int issued = 0;  // producer: tiles issued
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // A batch of tiles is issued with one warp instruction: lane l issues box
    // l (tile l / BPB; block, slab and K|V from l % BPB).  Block ids are
    // fetched a window of TPW tiles at a time (lane l holds block l % BPT of
    // tile l / BPT), double-buffered one window ahead so that table reads
    // never sit on the issue path.
    const int BPB = BPT * G_::kSlabs * 2;  // boxes per tile (<= 16)
    const int TPB = 32 / BPB;              // tiles per issue batch
    const int TPW = 32 / BPT;              // tiles per id window
    constexpr int kNoBlock = INT_MIN, kBadBlock = INT_MIN + 1;
    auto window_ids = [&](int w0) {
      const int t = w0 + lane / BPT;
      if (t >= len) return kNoBlock;
      const Cursor cu = locate(cum, B, NHG, start + t);
      const int lb = cu.j * BPT + lane % BPT;
      if (lb >= (ctxs[cu.s] + T - 1) / T) return kNoBlock;
      const int v = a.tables[static_cast<size_t>(cu.s) * a.max_blocks + lb];
      return (v >= 0 && v < a.num_blocks) ? v : kBadBlock;
    };
    int cur_ids = window_ids(0), nxt_ids = window_ids(TPW);
    int nb = 0;
    for (int k = 0; k < len; k += nb) {
      // A batch never holds more tiles than the ring, nor crosses an id
      // window.  Only its first slot is waited for; the tiles after it join
      // the batch if their slots are already free, so a released slot is
      // refilled at once instead of after the whole batch has drained.
      const int cap = min(min(TPB, len - k), min(NS, TPW - k % TPW));
      if (k > 0 && k % TPW == 0) {
        cur_ids = nxt_ids;
        nxt_ids = window_ids(k + TPW);
      }
      int n = 0;
      if (lane == 0) {
        bool ok = k < NS || mbar_wait(smem_u32(&empty[k % NS]), ((k / NS) - 1) & 1, kWaitNs);
        if (ok) {
          n = 1;
          while (n < cap && (k + n < NS ||
                             mbar_try_wait(smem_u32(&empty[(k + n) % NS]), (((k + n) / NS) - 1) & 1)))
            ++n;
        }
      }
      nb = __shfl_sync(FULL, n, 0);
      if (nb == 0) s_abort = 1;
      if (__shfl_sync(FULL, s_abort, 0)) break;

      // this lane's box: tile k + lane / BPB
      const int tt = lane / BPB, bx = lane % BPB;
      const int blk = bx / (G_::kSlabs * 2), sl = (bx / 2) % G_::kSlabs, isv = bx & 1;
      const int id = __shfl_sync(FULL, cur_ids, ((k + tt) % TPW) * BPT + blk);
      const bool mine = tt < nb;
      const unsigned okmask = __ballot_sync(FULL, mine && id >= 0);
      const unsigned badmask = __ballot_sync(FULL, mine && id == kBadBlock);
      // per-tile bookkeeping by lane i for tile k + i; the first two tiles of
      // a pair in this CTA also carry its q rows (one for each consumer group)
      Cursor cu{0, 0, 0, 1};
      if (lane < nb) cu = locate(cum, B, NHG, start + k + lane);
      const int t_local = k + lane;
      const bool with_q = lane < nb && (cu.j <= 1 || t_local <= 1);
      if (lane < nb) {
        const int slot = t_local % NS;
        const unsigned tmask = ((1u << BPB) - 1u) << (lane * BPB);
        sbad[slot] = (badmask & tmask) != 0;
        const uint32_t bytes = __popc(okmask & tmask) * box_bytes +
                               (with_q ? static_cast<uint32_t>(QROWS) * D * 2u : 0u);
        mbar_arrive_expect_tx(smem_u32(&full[slot]), bytes);
      }
      const int hg = __shfl_sync(FULL, cu.h, tt < nb ? tt : 0);
      __syncwarp();
      if (mine && id >= 0) {
        const int slot = (k + tt) % NS;
        const uint8_t* tile_base = ring + static_cast<size_t>(slot) * G_::kStageBytes +
                                   (isv ? G_::kTileBytes : 0);
        tma_load_2d(smem_u32(tile_base + sl * kHalfBytes + blk * box_bytes), isv ? &vmap : &kmap,
                    sl * 128, (id * NKV + hg * HG) * T, smem_u32(&full[slot]));
      }
      if (with_q) {
        const int slot = t_local % NS;
        const typename Q::raw* qsrc = static_cast<const typename Q::raw*>(a.q) +
                                      (static_cast<size_t>(cu.s) * a.num_q_heads +
                                       static_cast<size_t>(cu.h) * QROWS) * D;
        bulk_load(smem_u32(qbuf + static_cast<size_t>(slot) * QB), qsrc,
                  static_cast<uint32_t>(QROWS) * D * 2u, smem_u32(&full[slot]));
      }
      issued = k + nb;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, q4 = lane & 3;
    const int group = warp / kWarps, row0 = (warp % kWarps) * 16;
    // the warp's 16 tile rows: block row0 / box_rows of the tile, head
    // (row0 % box_rows) / T of the group, tokens from (row0 % T)
    const int my_head = (row0 % box_rows) / T;
    const int my_tok = (row0 / box_rows) * T + row0 % T;
    WarpState<D> st;
    st.reset();
    uint32_t qa[KS][4];
    Cursor cur = locate(cum, B, NHG, start);
    int seg_j0 = cur.j;
    bool first_seg = true, seg_bad = false, need_q = true;
    for (int k = 0; k < len; ++k) {
      const int s = cur.s, hg = cur.h, j = cur.j;
      if (k % kGroups == group && s_abort) {
        seg_bad = true;  // after a stall nothing more is waited for or released
      } else if (k % kGroups == group) {
        const int slot = k % NS;
        const bool arrived = mbar_wait(smem_u32(&full[slot]), (k / NS) & 1, kWaitNs);
        if (!arrived) {
          s_abort = 1;
          seg_bad = true;
        }
        uint8_t* kt = ring + static_cast<size_t>(slot) * G_::kStageBytes;
        uint8_t* vt = kt + G_::kTileBytes;
        if (need_q) {  // this group's first tile of the pair carries q
          load_q<KV, Q, D>(qa,
                           reinterpret_cast<const typename Q::raw*>(qbuf + static_cast<size_t>(slot) * QB) +
                               static_cast<size_t>(my_head) * G * D,
                           G, g, q4);
          need_q = false;
        }
        seg_bad |= sbad[slot] != 0;
        const int nvalid = min(16, ctxs[s] - (j * TOKS + my_tok));
        bool zeroed = false;
        if (arrived && nvalid > 0)
          zeroed = tile_step<KV, D>(st, qa, kt, vt, row0, nvalid, a.qk_scale, lane);
        if (zeroed) fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
      }

      const bool seg_last = j == cur.nt - 1 || k == len - 1;
      if (seg_last) {
        const bool complete = seg_j0 == 0 && j == cur.nt - 1;
        if (seg_bad) s_segbad = 1;
        publish<KV, D>(st, mS, lS, oS, warp, G, G, lane);
        consumer_sync();
        const bool bad = s_segbad != 0;
        const size_t head0 = static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(hg) * QROWS;
        float* part = a.ws_part + static_cast<size_t>(2 * c + (first_seg ? 0 : 1)) * PS;
        for (int i = tid; i < QROWS * D; i += kConsumerWarps * 32) {
          const int qr = i / D, d = i - qr * D;  // qr = head * G + row
          const int hh = qr / G, row = qr - hh * G;
          // the warps that hold head hh (both groups, every 16-token unit)
          float M = -CUDART_INF_F;
          for (int w = 0; w < kConsumerWarps; ++w)
            if ((((w % kWarps) * 16) % box_rows) / T == hh) M = fmaxf(M, mS[w * 16 + row]);
          float L = 0.f, A = 0.f;
          if (M != -CUDART_INF_F) {
            for (int w = 0; w < kConsumerWarps; ++w) {
              if ((((w % kWarps) * 16) % box_rows) / T != hh) continue;
              const float f = exp2f(mS[w * 16 + row] - M);
              L = fmaf(lS[w * 16 + row], f, L);
              A = fmaf(oS[(w * G + row) * D + d], f, A);
            }
          }
          if (complete) {
            const float o = bad ? CUDART_NAN_F : (L > 0.f ? A * a.v_scale / L : 0.f);
            store_elem<Q>(a.out, (head0 + qr) * D + d, o);
          } else {
            part[qr * (D + 2) + 2 + d] = bad ? CUDART_NAN_F : A;
            if (d == 0) {
              part[qr * (D + 2)] = M;
              part[qr * (D + 2) + 1] = bad ? CUDART_NAN_F : L;
            }
          }
        }
        if (!complete) __threadfence();
        consumer_sync();
        if (!complete) {
          const int P0 = cum[s] + hg * cur.nt;
          const int c0 = sp.owner(P0), c1 = sp.owner(P0 + cur.nt - 1);
          if (tid == 0) {
            const int prev = atomicAdd(&a.counters[static_cast<size_t>(s) * NHG + hg], 1);
            s_last = prev == c1 - c0;
          }
          consumer_sync();
          if (s_last) {
            __threadfence();
            for (int i = tid; i < QROWS * D; i += kConsumerWarps * 32) {
              const int qr = i / D, d = i - qr * D;
              float M = -CUDART_INF_F;
              for (int cc = c0; cc <= c1; ++cc) {
                const int which = cc == c0 ? (sp.start(cc) == P0 ? 0 : 1) : 0;
                M = fmaxf(M, __ldcg(a.ws_part + static_cast<size_t>(2 * cc + which) * PS +
                                    qr * (D + 2)));
              }
              float L = 0.f, A = 0.f;
              if (M != -CUDART_INF_F) {
                for (int cc = c0; cc <= c1; ++cc) {
                  const int which = cc == c0 ? (sp.start(cc) == P0 ? 0 : 1) : 0;
                  const float* pp =
                      a.ws_part + static_cast<size_t>(2 * cc + which) * PS + qr * (D + 2);
                  const float f = exp2f(__ldcg(pp) - M);
                  L = fmaf(__ldcg(pp + 1), f, L);
                  A = fmaf(__ldcg(pp + 2 + d), f, A);
                }
              }
              const float o = (L > 0.f || L != L) ? A * a.v_scale / L : 0.f;
              store_elem<Q>(a.out, (head0 + qr) * D + d, o);
            }
            if (tid == 0) atomicExch(&a.counters[static_cast<size_t>(s) * NHG + hg], 0);
          }
        }
        if (tid == 0) s_segbad = 0;
        consumer_sync();  // merge buffers and flags are free again
        st.reset();
        seg_bad = false;
        first_seg = false;
        need_q = true;
      }
      if (k + 1 < len) {
        advance(cur, cum, NHG);
        if (seg_last) seg_j0 = cur.j;
      }
    }
  }

  // ---- after a stall: wait (bounded) for the copies still in flight
  __syncthreads();
  if (s_abort && warp == kProducerWarp && lane == 0) {
    for (int k = max(0, issued - NS); k < issued; ++k)
      mbar_wait(smem_u32(&full[k % NS]), (k / NS) & 1, kDrainNs);
  }
}

}  // namespace tc

// Launch the persistent tensor-core decode kernel for one (cache, q) dtype pair.
template <typename KV, typename Q>
pkv_status launch_decode_persist(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pkv
