// The positions past a shared prefix, streamed by warps that each take
// (sequence, split, KV head) units from a queue.
//
// What it computes is the decode kernel's (attention_tc.cuh) for the
// positions [P, ctx) of every sequence behind a shared-prefix pass: for the G
// query heads of one KV head, the split's softmax partial (max, sum,
// unnormalised output) over its positions, K/V gathered through the block
// table (the katajob Q&A, "The paging idea"), written to the split's
// workspace slot for the merge kernel that follows.  Splits, tile order and
// arithmetic are the one-warp split form's, so the partials are the same
// values.
//
// Why a queue: past a shared prefix the contexts left are short (tens to a
// few hundred tokens), and a CTA per unit spends about as long reading its
// length, block ids and first tile, and writing its partial, as streaming
// its tiles; an SM whose CTAs drew short units runs dry while others finish
// long ones, and the SMs the pass holds at first get no unit at all once the
// grid has been handed out.  Here one CTA per SM runs twelve independent
// warps, each with its own two-stage TMA ring that it keeps streaming from
// one unit into the next, resolving the next unit (an atomic claim, its block
// ids and query rows) while the current one's last tiles are consumed; CTAs
// that become resident late (on the SMs the pass frees) take what is left.
// Units are handed out longest first: every CTA builds the same order from
// the batch's lengths (all its warps together, once), so that the last ones
// claimed are short and the SMs drain together.
//
// Bounded waits as in the decode kernel: a warp whose stage wait gives up
// sets the device error bit and turns every unit it holds or claims later
// into NaN partials (it issues no copy after it), after waiting, with its own
// bound, for its copies in flight.  A table entry out of range or a bad
// length makes that unit's partial NaN.  The queue counter and the grid's
// exit counter are reset by the last CTA to finish, which first waits for
// the pass's grid, so this grid completes after the pass.
#pragma once

#include "attention_tc.cuh"

namespace pkv {
namespace tc {

constexpr int kTailStages = 2;       // 8 KiB stages (16 tokens of K and of V) per warp
constexpr int kTailWarps = 12;       // streams per CTA, one CTA per SM
constexpr int kTailMaxTiles = 32;    // tiles of one unit: one block id per lane
constexpr int kTailBuckets = kTailMaxTiles + 1;  // unit sizes 0 .. 32 tiles
constexpr int kTailLead = 4;         // tiles before a unit's end at which the next is claimed
// Largest batch the per-CTA unit list covers (lengths, per-chunk size counts
// and units in shared memory): past it the one-warp split form runs instead.
constexpr int kTailMaxSeqs = 512;
constexpr int kTailMaxUnits = 1024;  // (sequence, split) entries
// A warp's partial goes out through shared memory, four heads at a time:
// rows of 132 floats (the padding keeps the fragment writes conflict-free).
constexpr int kTailStageHeads = 4;
constexpr int kTailStageRow = 132;

// Dynamic shared memory of the queue kernel (NW warps of NS stages) for a
// batch of B sequences and E (sequence, split) entries: the 1024-aligned
// rings, their barriers, the partial staging rows, the size counts per
// 32-sequence chunk, the bucket offsets, the lengths and the entries.
__host__ __device__ constexpr int tail_smem_bytes(int NW, int NS, int B, int E) {
  return 1024 + NW * NS * Geom<BF16, 128, 1>::kStageBytes + NW * NS * 8 +
         NW * kTailStageHeads * kTailStageRow * 4 + ((B + 31) / 32) * kTailBuckets * 4 +
         (kTailBuckets + 1) * 4 + 4 * B + 4 * E;
}

// One unit: a (sequence, split) entry of the list and a KV head.
struct TailUnit {
  int seq, kvh, split, t_begin, t_end, n_tiles, first_blk;
  int bad;      // PKV_DEVICE_* bits of this unit
  int bid;      // this lane's block id: the block of tile `lane`
  bool last;    // holds position ctx - 1 (the fused slot write)
};

// NW: warps (independent streams) per CTA; NS: ring stages per warp; LEAD:
// tiles before a unit's end at which the next unit is claimed (resolved one
// tile later).
template <typename KV, typename Q, int NW = kTailWarps, int NS = kTailStages, int LEAD = kTailLead>
__global__ void __launch_bounds__(32 * NW, 1)
    tail_stream_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  constexpr int D = 128, T = 16, NT = 32 * NW;
  using G_ = Geom<KV, D, 1>;
  constexpr uint32_t kBoxBytes = static_cast<uint32_t>(T * G_::kRowBytes);
  static_assert(G_::kTileBytes == kBoxBytes, "one block per tile");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q4 = lane & 3;
  if (tid < 2)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tid ? &vmap : &kmap))
                 : "memory");
  // the merge kernel after this grid may be scheduled once every CTA runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int P = a.prefix_tokens, B = a.num_seqs, NKV = a.num_kv_heads, G = a.group;
  const int E = B * (a.max_splits - a.prefix_splits);  // entry capacity
  const int n_chunks = (B + 31) / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = base + warp * NS * G_::kStageBytes;  // this warp's ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + NW * NS * G_::kStageBytes) + warp * NS;
  float* s_part_all = reinterpret_cast<float*>(base + NW * NS * G_::kStageBytes + NW * NS * 8);
  float* s_part = s_part_all + warp * kTailStageHeads * kTailStageRow;  // this warp's staging rows
  int* s_tab = reinterpret_cast<int*>(s_part_all + NW * kTailStageHeads * kTailStageRow);
  int* s_off = s_tab + n_chunks * kTailBuckets;  // bucket offsets, then the entry count
  int* s_ctx = s_off + kTailBuckets + 1;
  uint32_t* s_ent = reinterpret_cast<uint32_t*>(s_ctx + B);

  int* queue = a.done + 1;

  // ------------------------------------------------ the unit list, longest first
  // A sequence's positions past the prefix split as in the decode kernel:
  // n_t 16-token tiles shared out evenly over nsplit splits.
  auto geometry = [&](int ctx, int& n_t, int& ns) {
    const bool bad = ctx < 0 || ctx > a.max_blocks * T || ctx <= P;
    const int own = bad ? 0 : ctx - P;
    ns = bad ? 1 : max(1, (own + a.partition - 1) / a.partition);
    n_t = (own + T - 1) / T;
  };
  auto bucket_of = [&](int n_t, int ns, int i) {
    return min(kTailMaxTiles, (i + 1) * n_t / ns - i * n_t / ns);
  };
  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&bars[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  for (int i = tid; i < n_chunks * kTailBuckets; i += NT) s_tab[i] = 0;
  for (int s = tid; s < B; s += NT) s_ctx[s] = a.ctx_lens[s];
  __syncthreads();
  // size counts per 32-sequence chunk (warp w takes chunks w, w + NW, ...)
  for (int c = warp; c < n_chunks; c += NW) {
    const int s = 32 * c + lane;
    if (s < B) {
      int n_t, ns;
      geometry(s_ctx[s], n_t, ns);
      for (int i = 0; i < ns; ++i) atomicAdd(&s_tab[c * kTailBuckets + bucket_of(n_t, ns, i)], 1);
    }
  }
  __syncthreads();
  // each bucket's count over the chunks before (a column scan), its total
  for (int b = tid; b < kTailBuckets; b += NT) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int n = s_tab[c * kTailBuckets + b];
      s_tab[c * kTailBuckets + b] = run;
      run += n;
    }
    s_off[b] = run;
  }
  __syncthreads();
  if (tid == 0) {  // bucket offsets, largest units first; then the entry count
    int off = 0;
    for (int b = kTailBuckets - 1; b >= 0; --b) {
      const int n = s_off[b];
      s_off[b] = off;
      off += n;
    }
    s_off[kTailBuckets] = off;
  }
  __syncthreads();
  // Scatter: within a bucket, chunk by chunk, then by split index, then by
  // lane, so that every CTA builds the same list.
  for (int c = warp; c < n_chunks; c += NW) {
    const int s = 32 * c + lane;
    int n_t = 0, ns = 0;
    if (s < B) geometry(s_ctx[s], n_t, ns);
    int max_ns = ns;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) max_ns = max(max_ns, __shfl_xor_sync(0xffffffffu, max_ns, o));
    int* run = s_tab + c * kTailBuckets;  // this chunk's running positions within each bucket
    for (int i = 0; i < max_ns; ++i) {
      const bool has = i < ns;
      const int b = has ? bucket_of(n_t, ns, i) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, b);
      const int rank = __popc(peers & ((1u << lane) - 1));
      if (has) s_ent[s_off[b] + run[b] + rank] = (static_cast<uint32_t>(s) << 8) | static_cast<uint32_t>(i);
      __syncwarp();
      if (has && rank == 0) run[b] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  const int n_units = min(s_off[kTailBuckets], E) * NKV;

  // ------------------------------------------------ units
  // Claim index k -> entry k / N_kv (longest first), KV head k % N_kv.
  auto resolve = [&](int k, TailUnit& u) {
    const uint32_t ent = s_ent[k / NKV];
    u.seq = static_cast<int>(ent >> 8);
    u.split = static_cast<int>(ent & 255u);
    u.kvh = k % NKV;
    const int ctx = s_ctx[u.seq];
    int n_t, ns;
    geometry(ctx, n_t, ns);
    const bool bad = ctx < 0 || ctx > a.max_blocks * T || ctx <= P;
    u.bad = bad ? kBadLength : 0;
    const int tb = u.split * n_t / ns, te = (u.split + 1) * n_t / ns;
    u.t_begin = P + tb * T;
    u.t_end = bad ? u.t_begin : min(P + te * T, ctx);
    u.n_tiles = bad ? 0 : te - tb;
    u.first_blk = u.t_begin / T;
    u.last = !bad && ctx > 0 && u.split == ns - 1;
    const int32_t* trow = a.tables + static_cast<size_t>(u.seq) * a.max_blocks;
    u.bid = lane < u.n_tiles ? trow[u.first_blk + lane] : -1;
  };
  const typename Q::raw* q_base = static_cast<const typename Q::raw*>(a.q);
  auto load_query = [&](uint32_t (&qb)[D / 16][2], const TailUnit& u) {
    load_qt<KV, Q, D>(qb, q_base + (static_cast<size_t>(u.seq) * a.num_q_heads +
                                    static_cast<size_t>(u.kvh) * G) * D, G, g, q4);
  };
  const HeadScales sc0 = head_scales(a.head_scales, NKV, 0, a.softmax_scale, a.qk_scale, a.v_scale,
                                     a.k_inv, a.v_inv);

  // The step's token of a unit holding position ctx - 1, written before any
  // of its copies is issued (no other unit reads that row of the block).
  auto slot_write = [&](const TailUnit& u) {
    if (a.k_new == nullptr || !u.last) return;
    const int p = s_ctx[u.seq] - 1;
    const int blk = __shfl_sync(0xffffffffu, u.bid, (p / T - u.first_blk) & 31);
    if (blk >= 0 && blk < a.num_blocks) {
      const int which = lane / 16, d0 = (lane % 16) * 8;
      const size_t src = (static_cast<size_t>(u.seq) * NKV + u.kvh) * D + d0;
      const size_t dst = ((static_cast<size_t>(blk) * NKV + u.kvh) * T + p % T) * D + d0;
      store8<Q, KV>(static_cast<const typename Q::raw*>(which ? a.v_new : a.k_new) + src,
                    static_cast<typename KV::raw*>(const_cast<void*>(which ? a.v_cache : a.k_cache)) + dst,
                    which ? sc0.v_inv : sc0.k_inv);
      asm volatile("fence.proxy.async.global;" ::: "memory");  // before the TMA reads it
    }
    __syncwarp();
  };

  // Issue tile `t` of unit u into ring slot `ki`: lane 0 the K box, lane 1
  // the V box.  Returns the unit's new bad bits.
  auto issue = [&](const TailUnit& u, int t, int ki) {
    const int s = ki % NS;
    const int phys = __shfl_sync(0xffffffffu, u.bid, t);
    const bool good = phys >= 0 && phys < a.num_blocks;
    const uint32_t bar = smem_u32(&bars[s]);
    if (lane == 0) mbar_arrive_expect_tx(bar, good ? 2 * kBoxBytes : 0);
    __syncwarp();
    if (good && lane < 2) {
      uint8_t* dst = stages + s * G_::kStageBytes + (lane ? G_::kTileBytes : 0);
      tma_box<KV, D>(smem_u32(dst), lane ? &vmap : &kmap, (phys * NKV + u.kvh) * T, bar);
    }
    return good ? 0 : kBadTable;
  };

  // The partial of a unit from the warp's state: the one-warp split form's
  // warp merge with a single warp (M = m, L = l, A = o, or 0 and 0 where no
  // position was attended), A times the V scale.
  auto write_partial = [&](const WarpStateT<D>& st, const TailUnit& u, bool bad) {
    const HeadScales sc = head_scales(a.head_scales, NKV, u.kvh, a.softmax_scale, a.qk_scale,
                                      a.v_scale, a.k_inv, a.v_inv);
    const size_t head0 = static_cast<size_t>(u.seq) * a.num_q_heads + static_cast<size_t>(u.kvh) * G;
    float M[2], L[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = st.l[j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      M[j] = st.m[j];
      L[j] = M[j] != -CUDART_INF_F ? fmaf(l, exp2f(M[j] - M[j]), 0.f) : 0.f;
      const int head = 2 * q4 + j;
      if (g == 0 && head < G) {
        const size_t pidx = (head0 + head) * a.max_splits + u.split;
        a.ws_m[pidx] = M[j];
        a.ws_l[pidx] = bad ? CUDART_NAN_F : L[j];
      }
    }
    // the outputs, four heads at a time: fragments into the staging rows,
    // then whole 512-byte rows out with 16-byte stores
#pragma unroll
    for (int h0 = 0; h0 < 8; h0 += kTailStageHeads) {
      if (h0 >= G) break;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = e & 1, head = 2 * q4 + j;
          if (head >= h0 && head < h0 + kTailStageHeads) {
            float A = M[j] != -CUDART_INF_F ? fmaf(st.o[mt][e], exp2f(M[j] - M[j]), 0.f) : 0.f;
            A *= sc.v;
            s_part[(head - h0) * kTailStageRow + out_row_t<false>(mt, g, e >> 1)] = bad ? CUDART_NAN_F : A;
          }
        }
      __syncwarp();
      const int nh = min(kTailStageHeads, G - h0);
      for (int i = lane; i < nh * (D / 4); i += 32) {
        const int hl = i / (D / 4), c4 = i % (D / 4);
        const size_t pidx = (head0 + h0 + hl) * a.max_splits + u.split;
        reinterpret_cast<float4*>(a.ws_acc + pidx * D)[c4] =
            *reinterpret_cast<const float4*>(s_part + hl * kTailStageRow + 4 * c4);
      }
      __syncwarp();
    }
  };

  // ------------------------------------------------ stream
  int claim = 0;
  if (lane == 0) claim = atomicAdd(queue, 1);
  claim = __shfl_sync(0xffffffffu, claim, 0);
  int warp_bits = 0;
  if (claim < n_units) {
    TailUnit cur, nxt;
    resolve(claim, cur);
    uint32_t qb[D / 16][2], qn[D / 16][2];
    load_query(qb, cur);
    // next unit: 0 = not claimed, 1 = claim in flight, 2 = resolved, 3 = none left
    int ns_state = 0;
    int ki = 0, kc = 0;          // ring slots issued / consumed by this warp
    int p_unit = 0, p_tile = 0;  // the producer: unit (0 cur, 1 nxt) and its next tile
    bool cur_started = false, nxt_started = false;
    bool failed = false;
    // issue the next tile in stream order if a slot is free and the tile known
    auto issue_next = [&]() -> bool {
      if (failed || ki >= kc + NS) return false;
      if (p_unit == 0 && p_tile >= cur.n_tiles) {
        if (ns_state != 2) return false;
        p_unit = 1;
        p_tile = 0;
      }
      TailUnit& u = p_unit == 0 ? cur : nxt;
      bool& started = p_unit == 0 ? cur_started : nxt_started;
      if (p_tile >= u.n_tiles) return false;
      if (!started) {
        slot_write(u);
        started = true;
      }
      u.bad |= issue(u, p_tile, ki);
      ++p_tile;
      ++ki;
      return true;
    };
    auto step_claims = [&](int remaining) {
      if (ns_state == 0 && remaining <= LEAD) {
        if (lane == 0) claim = atomicAdd(queue, 1);
        ns_state = 1;
      } else if (ns_state == 1) {
        const int k = __shfl_sync(0xffffffffu, claim, 0);
        if (k < n_units) {
          resolve(k, nxt);
          load_query(qn, nxt);
          nxt_started = false;
          ns_state = 2;
        } else {
          ns_state = 3;
        }
      }
    };
    while (issue_next()) {}

    WarpStateT<D> st;
    while (true) {
      st.reset();
      const HeadScales sc = head_scales(a.head_scales, NKV, cur.kvh, a.softmax_scale, a.qk_scale,
                                        a.v_scale, a.k_inv, a.v_inv);
      for (int t = 0; t < cur.n_tiles && !failed; ++t) {
        step_claims(cur.n_tiles - t);
        const int s = kc % NS;
        const bool arrived = stage_wait(smem_u32(&bars[s]), (kc / NS) & 1, a.wait_ns);
        if (!__all_sync(0xffffffffu, arrived)) {
          failed = true;
          break;
        }
        uint8_t* kt = stages + s * G_::kStageBytes;
        const int tok0 = cur.t_begin + t * T;
        const int nvalid = min(T, cur.t_end - tok0);
        const bool zeroed = tile_step_t<KV, D>(st, qb, kt, kt + G_::kTileBytes, 0, nvalid, sc.qk, lane);
        if (zeroed) fence_proxy_async();  // the zeroed rows, before the slot is refilled by TMA
        __syncwarp();
        ++kc;
        while (issue_next()) {}
      }
      if (failed) {
        // the copies still in flight land before the warp's ring goes
        if (lane == 0)
          for (int k = kc; k < ki; ++k) mbar_wait(smem_u32(&bars[k % NS]), (k / NS) & 1, kDrainNs);
        ki = kc;
        warp_bits |= kTimeout;
      }
      __syncwarp();
      warp_bits |= cur.bad;
      write_partial(st, cur, failed || cur.bad != 0);
      // the next unit: claimed and resolved now if the current one was short
      while (ns_state == 0 || ns_state == 1) step_claims(0);
      if (ns_state == 3) break;
      // rotate
      cur = nxt;
      cur_started = nxt_started;
  #pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qb[ks][0] = qn[ks][0];
        qb[ks][1] = qn[ks][1];
      }
      if (p_unit == 1) {
        p_unit = 0;
      } else {
        p_tile = 0;
      }
      ns_state = 0;
      while (issue_next()) {}
    }
  }
  // the warps' error bits, then the CTA counts out; the last CTA of the grid
  // waits for the pass's grid and resets the counters
  if (lane == 0 && warp_bits != 0 && a.status != nullptr) atomicOr(a.status, warp_bits);
  __syncthreads();
  if (tid == 0) {
    const int total = static_cast<int>(gridDim.x);
    if (atomicAdd(a.done, 1) == total - 1) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicExch(queue, 0);
      atomicExch(a.done, 0);
    }
  }
}

}  // namespace tc
}  // namespace pkv
