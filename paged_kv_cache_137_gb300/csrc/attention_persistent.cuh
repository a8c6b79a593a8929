// Persistent decode attention: a grid of resident CTAs that take work units
// (sequence, KV head, split) from a queue until it is empty.
//
// What it computes is the split kernel's (attention_tc.cuh): for the G query
// heads of one KV head, softmax(q . K^T * scale) V over the positions of one
// split, K/V gathered through the block table (the katajob Q&A, "The paging
// idea"; the foundry page on paged block allocation, "Concept"), the splits
// merged by the last to finish.
//
// Why a second schedule: when the units are short (a few 64-token tiles, as
// the private tails of sequences that share a prompt), a CTA per unit spends
// most of its life outside the stream of K/V: reading the length, then the
// block table, then waiting for the first tile, and at the end combining its
// warps and counting itself in, each a global round trip that costs several
// microseconds while HBM is saturated.  Here a CTA lives for the whole call:
//  * Every CTA numbers the units the same way (sequence by sequence, the
//    splits of a sequence, then its KV heads) from the lengths, which it
//    reads once into shared memory with a prefix sum of the units per
//    sequence.  A CTA takes the next unit number from a global counter one
//    unit ahead of need.
//  * Warp 0 resolves a unit ahead of the consumers: its block ids, the G
//    query rows and (for the step's token) the new K/V rows are copied into a
//    shared-memory slot by cp.async, with no thread waiting on them.  Two
//    slots: the unit being consumed and the next one.
//  * The K/V ring (two 32 KiB stages for 16-bit head_dim 128, three CTAs
//    per SM) is refilled across unit boundaries: the next unit's first tiles
//    are in flight while the current unit finishes.
//  * The tile math is the split kernel's (head-columns form, query groups of
//    up to 8): each warp folds 16 tokens of a tile into its own running
//    state, with one CTA barrier per tile.  At a unit's end the warps' states
//    are combined through the stage buffer of the unit's last tile, which is
//    handed back to the producer only after that; the other stage keeps the
//    next unit's first tile in flight.
//  * Split partials are counted in at the end of the CTA's life (or when 64
//    are pending): one fence, one atomic per unit, and the last of a pair's
//    partials to arrive merges them.  With a shared prefix the prefix pass's
//    partials join the same count.
//  * Every wait is bounded; a CTA whose stage wait gives up drains its copies
//    in flight, stops issuing, and finishes every unit it takes from then on
//    (including the rest of the queue, if no other CTA does) with NaN.
#pragma once

#include "attention_tc.cuh"

namespace pkv {
namespace tc {
namespace pd {

constexpr int kCtasPerSm = 3;
constexpr int kRingBytes = 65536;   // K/V stages per CTA
constexpr int kMaxSeqs = kPdMaxSeqs;        // sequences a call may hold (schedule in shared memory)
constexpr int kUnitBlocks = kPdUnitBlocks;  // block ids of one unit (a partition of at most 128 blocks)
constexpr int kDefer = 64;          // partials counted in at once

template <typename KV, int D>
constexpr int stages() {
  return kRingBytes / Geom<KV, D>::kStageBytes;
}

// A resolved unit.
struct Unit {
  int seq, kvh, split, nsplit;
  int t_begin, t_end, n_tiles, first_blk;
  int n_blk, flags, bad, ctx;
};
constexpr int kValid = 1, kEnd = 2, kWrite = 4;

// Shared-memory layout (bytes from the 1024-aligned base).
template <typename KV, int D>
struct Layout {
  static constexpr int kStage = Geom<KV, D>::kStageBytes;
  static constexpr int kSlotTab = kUnitBlocks * 4;          // int32 block ids
  static constexpr int kSlotQ = 8 * D * 2;                  // up to 8 query rows (16-bit)
  static constexpr int kSlotNew = 2 * D * 2;                // the step's K and V rows
  static constexpr int kSlot = kSlotTab + kSlotQ + kSlotNew;
  static constexpr int ring = 0;
  static constexpr int slots = ring + stages<KV, D>() * kStage;
  static constexpr int ctx = slots + 2 * kSlot;             // int32 [kMaxSeqs]
  static constexpr int cum = ctx + kMaxSeqs * 4;            // int32 [kMaxSeqs + 1], padded
  static constexpr int units = cum + (kMaxSeqs + 4) * 4;    // Unit [2]
  static constexpr int defer = units + 2 * static_cast<int>(sizeof(Unit));  // int4 [kDefer]
  static constexpr int bars = defer + kDefer * 16;          // uint64 [stages], then [2] slot ready
  static constexpr int bytes = bars + (stages<KV, D>() + 2) * 8 + 1024;  // + base alignment
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// The mbarrier at bar counts one arrival from this thread once all its
// cp.async copies issued so far have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

template <typename KV, typename Q, int D, int T>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_pd_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
  static_assert(!std::is_same<KV, E4M3>::value, "16-bit caches");
  static_assert(std::is_same<KV, Q>::value, "16-bit caches take queries of their own type");
  using G_ = Geom<KV, D>;
  using L_ = Layout<KV, D>;
  using raw = typename KV::raw;
  constexpr int NS = stages<KV, D>();
  constexpr int KS = D / 16;          // k-steps of S^T = K q^T
  constexpr int BPT = kTile / T;      // blocks per tile
  constexpr int BPB = BPT * 2;        // TMA boxes per tile (K and V of each block)
  constexpr int kBoxBytes = T * G_::kRowBytes;
  constexpr bool kBf = std::is_same<KV, BF16>::value;
  constexpr unsigned FULL = 0xffffffffu;
  static_assert(NS >= 2 && BPB <= 32, "ring and box lanes");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3, li = lane & 7, mi = lane >> 3;
  const int P = a.prefix_tokens;
  // Launched as a programmatic dependent of the previous kernel: nothing it
  // may write is read before it has completed.  Behind the shared-prefix
  // pass (which waited for everything before it before letting this grid
  // start) there is nothing to wait for: the pass's partials meet this
  // grid's through the arrival counters.
  if (P == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int B = a.num_seqs, NKV = a.num_kv_heads, G = a.group, HQ = a.num_q_heads;
  const int max_ctx = a.max_blocks * T;
  const int n_extra = P > 0 ? a.prefix_splits : 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem + L_::ring;
  int* s_ctx = reinterpret_cast<int*>(smem + L_::ctx);
  int* s_cum = reinterpret_cast<int*>(smem + L_::cum);
  Unit* s_unit = reinterpret_cast<Unit*>(smem + L_::units);
  int4* s_defer = reinterpret_cast<int4*>(smem + L_::defer);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L_::bars);
  uint64_t* s_ready = s_bar + NS;  // per slot: the resolved unit's copies have landed (32 arrivals)
  auto slot_tab = [&](int s) { return reinterpret_cast<int32_t*>(smem + L_::slots + s * L_::kSlot); };
  auto slot_q = [&](int s) {
    return reinterpret_cast<raw*>(smem + L_::slots + s * L_::kSlot + L_::kSlotTab);
  };
  auto slot_new = [&](int s) {
    return reinterpret_cast<raw*>(smem + L_::slots + s * L_::kSlot + L_::kSlotTab + L_::kSlotQ);
  };
  __shared__ int s_wsum[kWarps];
  __shared__ int s_ndefer, s_nlast, s_last[kDefer];

  // ------------------------------------------------------------ schedule
  // The units of sequence i: nsplit_i splits x N_kv heads, numbered sequence
  // by sequence; s_cum[i] = units before sequence i.
  auto nsplit_of = [&](int c) {
    const bool bad = c < 0 || c > max_ctx || (P > 0 && c <= P);
    return bad ? 1 : max(1, (c - P + a.partition - 1) / a.partition);
  };
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&s_bar[s]), 1);
    for (int s = 0; s < 2; ++s) mbar_init(smem_u32(&s_ready[s]), 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_ndefer = 0;
  }
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int run = 0;
    for (int i = b0; i < b1; ++i) {
      const int c = a.ctx_lens[i];
      s_ctx[i] = c;
      run += nsplit_of(c) * NKV;
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
    for (int i = b0; i < b1; ++i) {
      s_cum[i] = excl;
      excl += nsplit_of(s_ctx[i]) * NKV;
    }
    if (tid == kThreads - 1) s_cum[B] = excl;
    __syncthreads();
  }
  const int U = s_cum[B];

  // ------------------------------------------------- unit resolution (warp 0)
  // Unit v into slot s: geometry from the lengths, then the block ids, the
  // query rows and the step's K/V rows copied into the slot by cp.async.
  auto resolve = [&](int s, int v) {
    Unit u{};
    if (v >= U) {
      u.flags = kEnd;
    } else {
      int lo = 0, hi = B;  // s_cum[lo] <= v < s_cum[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_cum[mid] <= v) lo = mid;
        else hi = mid;
      }
      const int r = v - s_cum[lo];
      u.seq = lo;
      u.split = r / NKV;
      u.kvh = r - u.split * NKV;
      const int c = s_ctx[lo];
      const bool bad = c < 0 || c > max_ctx || (P > 0 && c <= P);
      const int own = bad ? 0 : c - P;
      u.nsplit = nsplit_of(c);
      const int n_t = (own + kTile - 1) / kTile;
      u.t_begin = P + (u.split * n_t / u.nsplit) * kTile;
      u.t_end = bad ? P : min(P + ((u.split + 1) * n_t / u.nsplit) * kTile, c);
      u.first_blk = u.t_begin / T;
      u.n_blk = (u.t_end - u.t_begin + T - 1) / T;
      u.n_tiles = (u.t_end - u.t_begin + kTile - 1) / kTile;
      u.bad = bad ? kBadLength : 0;
      u.ctx = c;
      const bool write = a.k_new != nullptr && !bad && c > 0 && u.split == u.nsplit - 1;
      u.flags = kValid | (write ? kWrite : 0);
      int32_t* tab = slot_tab(s);
      const int32_t* src = a.tables + static_cast<size_t>(u.seq) * a.max_blocks + u.first_blk;
      for (int i = lane; i < u.n_blk; i += 32) cp_async4(tab + i, src + i);
      const raw* qsrc = static_cast<const raw*>(a.q) + (static_cast<size_t>(u.seq) * HQ + u.kvh * G) * D;
      raw* qdst = slot_q(s);
      for (int i = lane; i < G * D / 8; i += 32) cp_async16(qdst + 8 * i, qsrc + 8 * i);
      if (write) {
        const size_t row = (static_cast<size_t>(u.seq) * NKV + u.kvh) * D;
        raw* ndst = slot_new(s);
        for (int i = lane; i < 2 * D / 8; i += 32)
          cp_async16(ndst + 8 * i, static_cast<const raw*>(i < D / 8 ? a.k_new : a.v_new) + row + 8 * (i % (D / 8)));
      }
    }
    cp_async_arrive(smem_u32(&s_ready[s]));  // every lane: once its copies have landed
    if (lane == 0) s_unit[s] = u;
    __syncwarp();
  };
  // Unit k is in slot k & 1, the ((k >> 1) + 1)-th use of that slot.
  auto ready_parity = [](int k) { return static_cast<uint32_t>((k >> 1) & 1); };

  // ------------------------------------------------------- producer (warp 0)
  int pu = 0, ptile = 0, issued = 0, pstarted = -1;  // warp 0's view
  int released = 0;                                  // tiles consumed (all threads)
  int cu = 0;                                        // unit being consumed (all threads)
  bool dead = false;                                 // a stage wait gave up
  auto issue = [&](int s, const Unit& u, int tile) {
    const int st = issued % NS;
    uint8_t* kt = ring + st * L_::kStage;
    const int lb0 = tile * BPT;
    const int blk = lane / 2, isv = lane & 1;
    int phys = -1;
    bool inb = false;
    if (lane < BPB && lb0 + blk < u.n_blk) {
      inb = true;
      phys = slot_tab(s)[lb0 + blk];
    }
    const bool good = inb && phys >= 0 && phys < a.num_blocks;
    const unsigned okmask = __ballot_sync(FULL, good);
    const unsigned badmask = __ballot_sync(FULL, inb && !good);
    const uint32_t bar = smem_u32(&s_bar[st]);
    if (lane == 0) {
      if (badmask) s_unit[s].bad |= kBadTable;
      mbar_arrive_expect_tx(bar, __popc(okmask) * static_cast<uint32_t>(kBoxBytes));
    }
    __syncwarp();
    if (good)
      tma_box<KV, D>(smem_u32(kt + (isv ? G_::kTileBytes : 0) + blk * kBoxBytes), isv ? &vmap : &kmap,
                     (phys * NKV + u.kvh) * T, bar);
    ++issued;
  };
  // The step's token of the unit in slot s, written into the cache before any
  // of the unit's tiles is fetched (the unit that holds position ctx - 1).
  auto store_new = [&](int s, const Unit& u) {
    const int p = u.ctx - 1;
    const int blk = slot_tab(s)[p / T - u.first_blk];
    if (blk >= 0 && blk < a.num_blocks) {
      const size_t dst = ((static_cast<size_t>(blk) * NKV + u.kvh) * T + p % T) * D;
      for (int i = lane; i < 2 * D / 8; i += 32) {
        raw* cache = static_cast<raw*>(const_cast<void*>(i < D / 8 ? a.k_cache : a.v_cache));
        *reinterpret_cast<uint4*>(cache + dst + 8 * (i % (D / 8))) =
            *reinterpret_cast<const uint4*>(slot_new(s) + 8 * i);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // before the TMA reads it
    }
    __syncwarp();
  };
  // Issue tiles while a stage is free, in unit order, up to one unit ahead of
  // the consumers (two slots).
  auto pump = [&]() {
    while (!dead && issued < released + NS && pu <= cu + 1) {
      const int s = pu & 1;
      const Unit u = s_unit[s];
      if (u.flags & kEnd) break;
      if (pstarted != pu) {  // the unit's copies must have landed; its token is written first
        if (!__all_sync(FULL, mbar_try_wait(smem_u32(&s_ready[s]), ready_parity(pu)))) break;
        if (u.flags & kWrite) store_new(s, u);
        pstarted = pu;
      }
      if (ptile < u.n_tiles) {
        issue(s, s_unit[s], ptile);
        ++ptile;
      } else {
        ++pu;
        ptile = 0;
      }
    }
  };

  int next_v = 0;
  if (warp == 0) {
    int v0 = 0, v1 = 0;
    if (lane == 0) {
      v0 = atomicAdd(a.work, 1);
      v1 = atomicAdd(a.work, 1);
      next_v = atomicAdd(a.work, 1);
    }
    v0 = __shfl_sync(FULL, v0, 0);
    v1 = __shfl_sync(FULL, v1, 0);
    resolve(0, v0);
    resolve(1, v1);
    pump();
  }

  // q fragments (B operand of S^T = K q^T) and this warp's running state of
  // the current unit (its tokens of every tile)
  uint32_t qb[KS][2];
  WarpStateT<D> st;

  // ------------------------------------------------------- deferred counting
  // Pending partials (seq, kvh, nsplit) are counted in; where a pair's last
  // partial has arrived its partials are merged into the output.
  auto flush = [&]() {
    __threadfence();
    if (tid == 0) s_nlast = 0;
    __syncthreads();
    const int nd = s_ndefer;
    for (int i = tid; i < nd; i += kThreads) {
      const int4 d = s_defer[i];
      const int prev = atomicAdd(&a.counters[static_cast<size_t>(d.x) * NKV + d.y], 1);
      if (prev == d.z + n_extra - 1) s_last[atomicAdd(&s_nlast, 1)] = i;
    }
    __syncthreads();
    const int nl = s_nlast;
    if (nl > 0) {
      __threadfence();
      for (int e = tid; e < nl * G * D; e += kThreads) {
        const int4 d = s_defer[s_last[e / (G * D)]];
        const int head = (e / D) % G, dd = e % D;
        const int nsplit = d.z, np = nsplit + n_extra;
        const size_t base = (static_cast<size_t>(d.x) * HQ + d.y * G + head) * a.max_splits;
        auto slot = [&](int i) { return i < nsplit ? i : a.max_splits - n_extra + (i - nsplit); };
        float M = -CUDART_INF_F;
        for (int i = 0; i < np; ++i) M = fmaxf(M, __ldcg(a.ws_m + base + slot(i)));
        float Ls = 0.f, A = 0.f;
        if (M != -CUDART_INF_F) {
          for (int i = 0; i < np; ++i) {
            const float f = exp2f(__ldcg(a.ws_m + base + slot(i)) - M);
            Ls = fmaf(__ldcg(a.ws_l + base + slot(i)), f, Ls);
            A = fmaf(__ldcg(a.ws_acc + (base + slot(i)) * D + dd), f, A);
          }
        } else {
          for (int i = 0; i < np; ++i) Ls += __ldcg(a.ws_l + base + slot(i));
        }
        store_elem<Q>(a.out, (static_cast<size_t>(d.x) * HQ + d.y * G + head) * D + dd,
                      (Ls > 0.f || Ls != Ls) ? A / Ls : 0.f);
      }
      __syncthreads();
      for (int i = tid; i < nl; i += kThreads) {
        const int4 d = s_defer[s_last[i]];
        atomicExch(&a.counters[static_cast<size_t>(d.x) * NKV + d.y], 0);
      }
    }
    __syncthreads();
    if (tid == 0) s_ndefer = 0;
    __syncthreads();
  };

  __syncthreads();
  // ------------------------------------------------------------- consumers
  for (;;) {
    __syncthreads();
    const int s = cu & 1;
    const Unit u = s_unit[s];
    if (u.flags & kEnd) break;
    // this unit's copies (tables, queries, new token); then the producer can
    // start it if it has not yet
    if (!mbar_wait(smem_u32(&s_ready[s]), ready_parity(cu), kDrainNs)) dead = true;
    if (__syncthreads_or(dead)) dead = true;
    if (warp == 0) pump();
    {
      const raw* qrows = slot_q(s);
      load_qt<KV, Q, D>(qb, qrows, G, g, q4);
    }
    st.reset();
    const HeadScales sc = head_scales(a.head_scales, NKV, u.kvh, a.softmax_scale, a.qk_scale,
                                      a.v_scale, a.k_inv, a.v_inv);

    // the stage of the unit's last tile stays with the consumers for the
    // warp merge
    int held = -1;
    for (int tile = 0; tile < u.n_tiles && !dead; ++tile) {
      const int stg = released % NS;
      const bool arrived = stage_wait(smem_u32(&s_bar[stg]), (released / NS) & 1, a.wait_ns);
      const uint8_t* kt = ring + stg * L_::kStage;
      uint8_t* vt = ring + stg * L_::kStage + G_::kTileBytes;
      const int row0 = warp * 16;
      const int nvalid = min(16, u.t_end - (u.t_begin + tile * kTile + row0));
      bool zeroed = false;
      if (arrived && nvalid > 0) zeroed = tile_step_t<KV, D>(st, qb, kt, vt, row0, nvalid, sc.qk, lane);
      if (zeroed) fence_proxy_async();  // the zeroed rows, before the stage is refilled by TMA
      if (__syncthreads_or(!arrived)) {
        dead = true;
        break;
      }
      if (tile + 1 < u.n_tiles) {
        ++released;
        if (warp == 0) pump();
      } else {
        held = stg;
      }
    }

    if (dead) {
      // drain the copies still in flight before anything else touches the
      // ring; from now on no tile is issued or waited for
      if (warp == 0) {
        if (lane == 0)
          for (int t = released; t < issued; ++t)
            mbar_wait(smem_u32(&s_bar[t % NS]), (t / NS) & 1, kDrainNs);
        released = issued;
        // a unit taken but never started still writes its token (its copies
        // have landed or the wait for them gave up)
        if (pstarted < cu && (u.flags & kWrite)) {
          cp_async_wait_all();
          __syncwarp();
          store_new(s, u);
          pstarted = cu;
        }
      }
      __syncthreads();
    }

    // ---------------------------------------------------- finish the unit
    const int bad = u.bad | s_unit[s].bad | (dead ? kTimeout : 0);
    const bool direct = u.nsplit == 1 && P == 0;
    const size_t head0 = static_cast<size_t>(u.seq) * HQ + static_cast<size_t>(u.kvh) * G;
    if (held >= 0 && !dead) {
      // the warps' states combined in the held stage buffer: maxima and sums
      // [warp][16], outputs [warp][8 heads][D]
      float* mS = reinterpret_cast<float*>(ring + held * L_::kStage);
      float* lS = mS + kWarps * 16;
      float* oS = lS + kWarps * 16;
      publish_t<KV, D>(st, mS, lS, oS, warp, G, 8, lane);
      __syncthreads();
      for (int i = tid; i < G * D; i += kThreads) {
        const int row = i / D, d = i % D;
        float M, L, A;
        combine_warps(mS, lS, oS, kWarps, 8, row, d, D, M, L, A);
        A *= sc.v;
        if (direct) {
          store_elem<Q>(a.out, (head0 + row) * D + d, bad ? CUDART_NAN_F : (L > 0.f ? A / L : 0.f));
        } else {
          const size_t pidx = (head0 + row) * a.max_splits + u.split;
          a.ws_acc[pidx * D + d] = bad ? CUDART_NAN_F : A;
          if (d == 0) {
            a.ws_m[pidx] = M;
            a.ws_l[pidx] = bad ? CUDART_NAN_F : L;
          }
        }
      }
      fence_proxy_async();  // the generic writes into the stage, before TMA refills it
      __syncthreads();
      ++released;
      if (warp == 0) pump();
    } else {
      // nothing attended (an empty or invalid unit) or a wait gave up
      for (int i = tid; i < G * D; i += kThreads) {
        const int row = i / D, d = i % D;
        if (direct) {
          store_elem<Q>(a.out, (head0 + row) * D + d, bad ? CUDART_NAN_F : 0.f);
        } else {
          const size_t pidx = (head0 + row) * a.max_splits + u.split;
          a.ws_acc[pidx * D + d] = bad ? CUDART_NAN_F : 0.f;
          if (d == 0) {
            a.ws_m[pidx] = -CUDART_INF_F;
            a.ws_l[pidx] = bad ? CUDART_NAN_F : 0.f;
          }
        }
      }
    }
    if (tid == 0) {
      if (bad && a.status != nullptr) atomicOr(a.status, bad);
      if (!direct) s_defer[s_ndefer++] = make_int4(u.seq, u.kvh, u.nsplit, u.split);
    }
    // the slot is free: resolve the unit after next into it
    __syncthreads();
    if (warp == 0) {
      int v = next_v;
      if (lane == 0) next_v = atomicAdd(a.work, 1);
      v = __shfl_sync(FULL, v, 0);
      resolve(s, v);
    }
    ++cu;
    if (warp == 0) pump();
    if (s_ndefer >= kDefer) flush();
  }

  // -------------------------------------------------------------- finish
  flush();
  if (tid == 0) {
    const int total = static_cast<int>(gridDim.x);
    if (atomicAdd(a.done, 1) == total - 1) {
      // the last CTA: the shared-prefix pass (if any) is complete before
      // this grid is, and the queue counter starts from 0 next call
      if (P > 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicExch(a.work, 0);
      atomicExch(a.done, 0);
    }
  }
}

}  // namespace pd
}  // namespace tc
}  // namespace pkv
