// Launch of the shared-prefix pass: the tcgen05 attention pipeline of
// attention_prefill_umma.cuh in its shared-prefix form (kCasc), one CTA per
// (group of whole sequences filling up to 256 query rows, key range, KV head);
// and the merge kernel that follows the decode kernel on that path.
#include <atomic>

#include "attention_prefill_umma.cuh"

namespace pkv {

template <typename KV, typename Q>
pkv_status launch_shared_prefix_pass(const PrefillArgs& a, int block_size, int key_splits,
                                     const CUtensorMap& kmap, const CUtensorMap& vmap,
                                     cudaStream_t st) {
  constexpr int smem = tc::umma::smem_bytes<KV>();
  auto kernel = block_size == 16 ? tc::umma::prefill_umma_kernel<KV, Q, 16, true>
                                 : tc::umma::prefill_umma_kernel<KV, Q, 32, true>;
  static std::atomic<uint64_t> configured[2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("shared-prefix pass: cudaGetDevice", e);
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  std::atomic<uint64_t>& done = configured[block_size == 16 ? 0 : 1];
  if (!bit || !(done.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_fail("shared-prefix pass: cudaFuncSetAttribute", e);
    done.fetch_or(bit);
  }
  // each CTA: sp_seqs whole sequences (all their query heads of one KV head)
  const int groups = (a.num_seqs + a.sp_seqs - 1) / a.sp_seqs;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(groups, key_splits, a.num_kv_heads);
  cfg.blockDim = dim3(tc::umma::threads<KV>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, kmap, vmap);
  if (e != cudaSuccess) return cuda_fail("shared-prefix pass: launch", e);
  return check_launch("shared-prefix pass (tcgen05)");
}

// The merge after the decode kernel on the shared-prefix path: one CTA per
// (sequence, KV head) combines its G query heads' partials, the decode
// kernel's splits of the positions past the prefix (slots 0 .. nsplit - 1)
// then the pass's key ranges (the last prefix_splits slots), gathered into
// shared memory with one round trip (the decode kernel's merge_splits, so the
// sums are the fused merge's, value for value).  A programmatic dependent of
// the decode grid, which completes only after the pass.
constexpr int kMergeStage = 4096;  // floats of gathered partials; more fall back to direct loads

template <typename Q>
__global__ void __launch_bounds__(tc::kThreads) prefix_merge_kernel(const DecodeArgs a) {
  __shared__ __align__(16) float stage[kMergeStage];
  const int kvh = blockIdx.x, seq = blockIdx.y;
  const int P = a.prefix_tokens, n_extra = a.prefix_splits;
  // The lengths are read before the grid dependency wait: none of the three
  // kernels of the call writes them, and this grid starts only after every
  // decode CTA has started, hence after the pass has passed its own wait on
  // the work before the call.
  const int ctx = a.ctx_lens[seq];
  const bool bad = ctx < 0 || ctx > a.max_blocks * a.block_size || ctx <= P;
  const int nsplit = bad ? 1 : max(1, (ctx - P + a.partition - 1) / a.partition);
  const size_t head0 = static_cast<size_t>(seq) * a.num_q_heads + static_cast<size_t>(kvh) * a.group;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  tc::merge_splits<Q, 128, tc::kThreads>(a, head0, nsplit, a.max_splits - n_extra, n_extra, stage,
                                         kMergeStage);
}

template <typename Q>
pkv_status launch_prefix_merge(const DecodeArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.num_kv_heads, a.num_seqs);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, prefix_merge_kernel<Q>, a);
  if (e != cudaSuccess) return cuda_fail("shared-prefix merge: launch", e);
  return check_launch("shared-prefix merge");
}

template pkv_status launch_prefix_merge<BF16>(const DecodeArgs&, cudaStream_t);
template pkv_status launch_prefix_merge<F16>(const DecodeArgs&, cudaStream_t);

template pkv_status launch_shared_prefix_pass<BF16, BF16>(const PrefillArgs&, int, int,
                                                          const CUtensorMap&, const CUtensorMap&,
                                                          cudaStream_t);
template pkv_status launch_shared_prefix_pass<F16, F16>(const PrefillArgs&, int, int,
                                                        const CUtensorMap&, const CUtensorMap&,
                                                        cudaStream_t);
template pkv_status launch_shared_prefix_pass<E4M3, BF16>(const PrefillArgs&, int, int,
                                                          const CUtensorMap&, const CUtensorMap&,
                                                          cudaStream_t);
template pkv_status launch_shared_prefix_pass<E4M3, F16>(const PrefillArgs&, int, int,
                                                         const CUtensorMap&, const CUtensorMap&,
                                                         cudaStream_t);

}  // namespace pkv
