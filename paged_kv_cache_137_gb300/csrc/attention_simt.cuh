// CUDA-core paged decode attention (the general path: every cache dtype,
// head_dim 64/128, block_size 16/32, query groups up to 16).
//
// What it computes (katajob Q&A, "The paging idea": the kernel gathers keys and
// values through the block table instead of assuming contiguity; foundry page
// on paged block allocation, "Concept": a weighted sum over logically ordered
// positions):  for the query heads j of one KV head h,
//   o_j = sum_p softmax_p(q_j . K[p] * scale) V[p],  K[p] = K_pool[table[p / T]][h][p % T].
//
// Work split: one CTA per (split, KV head, sequence); a split is a fixed range
// of logical positions [split * P, (split + 1) * P), so results depend only on
// logical positions, never on which physical blocks hold them.  The CTA's four
// warps take the split's blocks round robin.  For a block, 32 / T lanes share
// one token in the q.k phase (each covers D * T / 32 elements and the partial
// dots are summed with shuffles); the lanes then split head_dim for p.V.  All
// the query heads of the KV head (G of them, padded to GM) are processed
// together, so each K/V element is read from memory once per CTA.  The online
// softmax keeps a running maximum and sum per head in fp32, in the log2
// domain (q is pre-multiplied by scale * log2(e)).  The warps' states are
// merged in shared memory; with more than one split the CTA writes its
// (max, sum, unnormalised output) and a merge kernel combines the splits.
//
// Tokens past the context end are masked out of the softmax and skipped in
// p.V, so whatever the unused slots of a block hold never reaches the output.
#pragma once

#include <math_constants.h>

#include "attention.h"
#include "device_common.cuh"

namespace pkv {

constexpr int kSimtWarps = 4;

template <typename KV, typename Q, int D, int T, int GM>
__global__ void __launch_bounds__(kSimtWarps * 32) decode_simt_kernel(const DecodeArgs a) {
  constexpr int TPT = 32 / T;  // lanes per token in the q.k phase
  constexpr int DQ = D / TPT;  // elements per lane in the q.k phase
  constexpr int DV = D / 32;   // elements per lane in the p.V phase
  constexpr int KCH = 8;       // elements per K load
  using raw = typename KV::raw;
  constexpr unsigned FULL = 0xffffffffu;

  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = a.group;
  const int ctx = a.ctx_lens[seq];
  const bool bad_ctx = ctx < 0 || ctx > a.max_blocks * T;
  const int nsplit = bad_ctx ? 1 : max(1, (ctx + a.partition - 1) / a.partition);
  if (split >= nsplit) return;
  const HeadScales sc = head_scales(a.head_scales, a.num_kv_heads, kvh, a.softmax_scale,
                                    a.qk_scale, a.v_scale, a.k_inv, a.v_inv);
  const int t_begin = split * a.partition;
  const int t_end = bad_ctx ? 0 : min(t_begin + a.partition, ctx);

  __shared__ float q_s[GM][D];
  __shared__ float m_s[kSimtWarps][GM];
  __shared__ float l_s[kSimtWarps][GM];
  __shared__ int bad_s;  // PKV_DEVICE_* bits
  // p_s lives during the block loop, acc_s after it
  __shared__ union {
    float p[kSimtWarps][T][GM];
    float acc[kSimtWarps][GM][D];
  } u_s;
  auto& p_s = u_s.p;
  auto& acc_s = u_s.acc;

  if (threadIdx.x == 0) bad_s = bad_ctx ? PKV_DEVICE_BAD_LENGTH : 0;
  for (int i = threadIdx.x; i < GM * D; i += blockDim.x) {
    const int j = i / D, d = i % D;
    float x = 0.f;
    if (j < G)
      x = load_elem<Q>(a.q, (static_cast<size_t>(seq) * a.num_q_heads + kvh * G + j) * D + d) *
          sc.qk;
    q_s[j][d] = x;
  }
  __syncthreads();

  float m[GM], lsum[GM], acc[GM][DV];
#pragma unroll
  for (int j = 0; j < GM; ++j) {
    m[j] = -CUDART_INF_F;
    lsum[j] = 0.f;
#pragma unroll
    for (int e = 0; e < DV; ++e) acc[j][e] = 0.f;
  }

  const int tok = lane % T, part = lane / T;
  const size_t head_stride = static_cast<size_t>(T) * D;
  const size_t block_stride = static_cast<size_t>(a.num_kv_heads) * head_stride;
  bool bad = false;
  const int first_blk = t_begin / T;
  const int end_blk = (t_end + T - 1) / T;
  for (int blk = first_blk + warp; blk < end_blk; blk += kSimtWarps) {
    const int phys = a.tables[static_cast<size_t>(seq) * a.max_blocks + blk];
    if (phys < 0 || phys >= a.num_blocks) {  // warp-uniform
      bad = true;
      break;
    }
    const size_t base = static_cast<size_t>(phys) * block_stride + kvh * head_stride;

    // q . k for this lane's token and slice of head_dim
    float s[GM];
#pragma unroll
    for (int j = 0; j < GM; ++j) s[j] = 0.f;
    const raw* kp = static_cast<const raw*>(a.k_cache) + base + static_cast<size_t>(tok) * D + part * DQ;
#pragma unroll
    for (int d0 = 0; d0 < DQ; d0 += KCH) {
      float kf[KCH];
      LoadF32<KV, KCH>::run(kp + d0, kf);
#pragma unroll
      for (int j = 0; j < GM; ++j)
#pragma unroll
        for (int e = 0; e < KCH; ++e) s[j] = fmaf(q_s[j][part * DQ + d0 + e], kf[e], s[j]);
    }
#pragma unroll
    for (int off = T; off < 32; off <<= 1)
#pragma unroll
      for (int j = 0; j < GM; ++j) s[j] += __shfl_xor_sync(FULL, s[j], off);

    // online softmax over the block's tokens
    const bool valid = blk * T + tok < t_end;
    float corr[GM];
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      const float sj = valid ? s[j] : -CUDART_INF_F;
      float bm = sj;
#pragma unroll
      for (int off = 1; off < T; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, off));
      const float mn = fmaxf(m[j], bm);  // finite: the block holds a valid token
      const float p = exp2f(sj - mn);
      float ps = p;
#pragma unroll
      for (int off = 1; off < T; off <<= 1) ps += __shfl_xor_sync(FULL, ps, off);
      corr[j] = exp2f(m[j] - mn);
      lsum[j] = lsum[j] * corr[j] + ps;
      m[j] = mn;
      if (part == 0) p_s[warp][tok][j] = p;
    }
#pragma unroll
    for (int j = 0; j < GM; ++j)
#pragma unroll
      for (int e = 0; e < DV; ++e) acc[j][e] *= corr[j];
    __syncwarp();

    // p . V, lanes split head_dim
    const raw* vp = static_cast<const raw*>(a.v_cache) + base + lane * DV;
    const int n_valid = min(T, t_end - blk * T);
    for (int t = 0; t < n_valid; ++t) {
      float vf[DV];
      LoadF32<KV, DV>::run(vp + static_cast<size_t>(t) * D, vf);
#pragma unroll
      for (int j = 0; j < GM; ++j) {
        const float pj = p_s[warp][t][j];
#pragma unroll
        for (int e = 0; e < DV; ++e) acc[j][e] = fmaf(pj, vf[e], acc[j][e]);
      }
    }
    __syncwarp();
  }
  if (bad && lane == 0) atomicOr(&bad_s, PKV_DEVICE_BAD_TABLE);
  __syncthreads();  // every warp is done with p_s before acc_s overwrites it

  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < GM; ++j) {
      m_s[warp][j] = m[j];
      l_s[warp][j] = lsum[j];
    }
  }
#pragma unroll
  for (int j = 0; j < GM; ++j)
#pragma unroll
    for (int e = 0; e < DV; ++e) acc_s[warp][j][lane * DV + e] = acc[j][e];
  __syncthreads();

  const bool any_bad = bad_s != 0;
  if (threadIdx.x == 0 && any_bad && a.status != nullptr) atomicOr(a.status, bad_s);
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int j = i / D, d = i % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, m_s[w][j]);
    float L = 0.f, A = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kSimtWarps; ++w) {
        const float f = exp2f(m_s[w][j] - M);
        L = fmaf(l_s[w][j], f, L);
        A = fmaf(acc_s[w][j][d], f, A);
      }
    }
    A *= sc.v;
    const int qh = kvh * G + j;
    if (nsplit == 1) {
      const float o = any_bad ? CUDART_NAN_F : (L > 0.f ? A / L : 0.f);
      store_elem<Q>(a.out, (static_cast<size_t>(seq) * a.num_q_heads + qh) * D + d, o);
    } else {
      const size_t pidx = (static_cast<size_t>(seq) * a.num_q_heads + qh) * a.max_splits + split;
      a.ws_acc[pidx * D + d] = any_bad ? CUDART_NAN_F : A;
      if (d == 0) {
        a.ws_m[pidx] = M;
        a.ws_l[pidx] = any_bad ? CUDART_NAN_F : L;
      }
    }
  }
}

template <typename KV, typename Q, int D, int T>
pkv_status launch_simt_dt(const DecodeArgs& a, int gm, cudaStream_t st) {
  const dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  const dim3 block(kSimtWarps * 32);
  switch (gm) {
    case 1: decode_simt_kernel<KV, Q, D, T, 1><<<grid, block, 0, st>>>(a); break;
    case 4: decode_simt_kernel<KV, Q, D, T, 4><<<grid, block, 0, st>>>(a); break;
    case 8: decode_simt_kernel<KV, Q, D, T, 8><<<grid, block, 0, st>>>(a); break;
    case 16: decode_simt_kernel<KV, Q, D, T, 16><<<grid, block, 0, st>>>(a); break;
    default: return fail(PKV_ERR_UNSUPPORTED, "query group larger than 16");
  }
  return check_launch("pkv_attention_decode (simt)");
}

template <typename KV, typename Q>
pkv_status launch_decode_simt(const DecodeArgs& a, int head_dim, int gm, cudaStream_t st) {
  const int T = a.block_size;
  if (head_dim == 128 && T == 16) return launch_simt_dt<KV, Q, 128, 16>(a, gm, st);
  if (head_dim == 128 && T == 32) return launch_simt_dt<KV, Q, 128, 32>(a, gm, st);
  if (head_dim == 64 && T == 16) return launch_simt_dt<KV, Q, 64, 16>(a, gm, st);
  if (head_dim == 64 && T == 32) return launch_simt_dt<KV, Q, 64, 32>(a, gm, st);
  return fail(PKV_ERR_UNSUPPORTED, "head_dim/block_size combination not compiled");
}

}  // namespace pkv
