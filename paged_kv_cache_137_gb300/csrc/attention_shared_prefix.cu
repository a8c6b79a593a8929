// Launch of the shared-prefix pass: the tcgen05 attention pipeline of
// attention_prefill_umma.cuh in its shared-prefix form (kCasc), one CTA per
// (group of whole sequences filling up to 256 query rows, key range, KV head).
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
