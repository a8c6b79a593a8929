// Launch wrapper of the tensor-core decode kernel (included by the
// per-dtype instantiation units).
#pragma once

#include <atomic>

#include "attention_persist.cuh"

namespace pkv {
namespace tc {

// Stages per CTA: 64 KiB of ring for every cache type (three CTAs per SM).
template <typename KV, int D>
constexpr int stages() {
  return Geom<KV, D>::kStageBytes >= 32768 ? 2 : 4;
}

template <typename KV, typename Q, int D, int T>
pkv_status launch_dt(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     cudaStream_t st) {
  constexpr int NS = stages<KV, D>();
  constexpr int smem = smem_bytes<KV, D, NS>();
  auto kernel = decode_tc_kernel<KV, Q, D, T, NS>;
  // the shared-memory opt-in is per device
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaGetDevice", e);
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaFuncSetAttribute", e);
    configured.fetch_or(bit);
  }
  const dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
  kernel<<<grid, kThreads, smem, st>>>(a, kmap, vmap);
  return check_launch("pkv_attention_decode (tensor core)");
}

// Persistent kernel: one CTA per SM (at most kPersistMaxCtas), as many ring
// slots as the opt-in shared memory allows (2..8).
template <typename KV, typename Q, int D, int T>
pkv_status launch_persist_dt(DecodeArgs a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t st) {
  auto kernel = decode_persist_kernel<KV, Q, D, T>;
  int dev = 0, sms = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode (device query)", e);
  const int smem_max = optin - static_cast<int>(fa.sharedSizeBytes);  // dynamic part
  // The ring depth is a multiple of the consumer-group count, so that every
  // slot is always consumed by the same group and each parity wait targets
  // the next phase of its barrier (the producer clamps its batches to it).
  constexpr int kMinStages = kGroups;
  const int qrows = a.hg * a.group;
  int ns = kPersistMaxStages / kGroups * kGroups;
  while (ns > kMinStages && persist_smem_bytes(Geom<KV, D>::kStageBytes, D, ns, a.num_seqs,
                                               a.group, qrows) > static_cast<size_t>(smem_max))
    ns -= kGroups;
  const size_t smem =
      persist_smem_bytes(Geom<KV, D>::kStageBytes, D, ns, a.num_seqs, a.group, qrows);
  if (smem > static_cast<size_t>(smem_max))
    return fail(PKV_ERR_UNSUPPORTED, "persistent kernel: shared memory too small for this batch");
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaFuncSetAttribute", e);
    configured.fetch_or(bit);
  }
  a.stages = ns;
  const int ctas = sms < kPersistMaxCtas ? sms : kPersistMaxCtas;
  kernel<<<ctas, kPersistThreads, smem, st>>>(a, kmap, vmap);
  return check_launch("pkv_attention_decode (persistent)");
}

}  // namespace tc

template <typename KV, typename Q>
pkv_status launch_decode_persist(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t st) {
  const int T = a.block_size;
  if constexpr (std::is_same<KV, E4M3>::value) {
    if (head_dim == 128 && T == 16) return tc::launch_persist_dt<KV, Q, 128, 16>(a, kmap, vmap, st);
    if (head_dim == 128 && T == 32) return tc::launch_persist_dt<KV, Q, 128, 32>(a, kmap, vmap, st);
  } else {
    if (head_dim == 128 && T == 16) return tc::launch_persist_dt<KV, Q, 128, 16>(a, kmap, vmap, st);
    if (head_dim == 128 && T == 32) return tc::launch_persist_dt<KV, Q, 128, 32>(a, kmap, vmap, st);
    if (head_dim == 64 && T == 16) return tc::launch_persist_dt<KV, Q, 64, 16>(a, kmap, vmap, st);
    if (head_dim == 64 && T == 32) return tc::launch_persist_dt<KV, Q, 64, 32>(a, kmap, vmap, st);
  }
  return fail(PKV_ERR_UNSUPPORTED, "persistent kernel: head_dim/block_size not compiled");
}

template <typename KV, typename Q>
pkv_status launch_decode_tc(const DecodeArgs& a, int head_dim, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, cudaStream_t st) {
  const int T = a.block_size;
  if constexpr (std::is_same<KV, E4M3>::value) {
    if (head_dim == 128 && T == 16) return tc::launch_dt<KV, Q, 128, 16>(a, kmap, vmap, st);
    if (head_dim == 128 && T == 32) return tc::launch_dt<KV, Q, 128, 32>(a, kmap, vmap, st);
  } else {
    if (head_dim == 128 && T == 16) return tc::launch_dt<KV, Q, 128, 16>(a, kmap, vmap, st);
    if (head_dim == 128 && T == 32) return tc::launch_dt<KV, Q, 128, 32>(a, kmap, vmap, st);
    if (head_dim == 64 && T == 16) return tc::launch_dt<KV, Q, 64, 16>(a, kmap, vmap, st);
    if (head_dim == 64 && T == 32) return tc::launch_dt<KV, Q, 64, 32>(a, kmap, vmap, st);
  }
  return fail(PKV_ERR_UNSUPPORTED, "tensor-core kernel: head_dim/block_size not compiled");
}

}  // namespace pkv
