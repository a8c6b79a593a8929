// Launch wrapper of the tensor-core decode kernel (included by the
// per-dtype instantiation units).
#pragma once

#include <algorithm>
#include <atomic>
#include <utility>

#include "attention_tail.cuh"

namespace pkv {
namespace tc {

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel in the stream drains; the kernel itself waits
// (griddepcontrol.wait) before reading its inputs.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, int threads, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Stages per CTA: 64 KiB of ring at three CTAs per SM (2 x 32 KiB or
// 4 x 16 KiB), 48 KiB (3 x 16 KiB) at four; the narrow forms two stages of
// their 8 or 16 KiB tiles.
template <typename KV, int D, bool HC, int W>
constexpr int stages() {
  if (W <= 2) return 2;
  if (Geom<KV, D>::kStageBytes >= 32768) return 2;
  return split_ctas_per_sm<KV, HC>() == 4 ? 3 : 4;
}

template <typename KV, typename Q, int D, int T, bool HC, int W = kWarps>
pkv_status launch_form(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       cudaStream_t st) {
  constexpr int NS = stages<KV, D, HC, W>();
  constexpr int smem = smem_bytes<KV, D, NS, W>();
  auto kernel = decode_tc_kernel<KV, Q, D, T, NS, HC, W>;
  // the shared-memory opt-in is per device
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaGetDevice", e);
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaFuncSetAttribute", e);
    configured.fetch_or(bit);
  }
  // the last prefix_splits split slots belong to the shared-prefix pass
  const dim3 grid(a.num_kv_heads, a.num_seqs, a.max_splits - (a.prefix_tokens > 0 ? a.prefix_splits : 0));
  e = launch_dependent(kernel, grid, 32 * W, smem, st, a, kmap, vmap);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: launch", e);
  return check_launch("pkv_attention_decode (tensor core)");
}

// The queue form of the positions past a shared prefix (attention_tail.cuh),
// for 16-bit head_dim-128 caches at block size 16 with units of at most 32
// tiles and a batch whose unit list fits its shared memory: one CTA of NW
// streaming warps per resident slot (one per SM).  Returns
// PKV_ERR_UNSUPPORTED (nothing launched, no error recorded) where it does
// not apply.
template <typename KV, typename Q, int NW = kTailWarps, int NS = kTailStages, int LEAD = kTailLead>
pkv_status launch_tail(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       cudaStream_t st) {
  const int tail_splits = a.max_splits - a.prefix_splits;
  const int64_t entries = static_cast<int64_t>(a.num_seqs) * tail_splits;
  if (a.group > 8 || a.partition / 16 > kTailMaxTiles || a.num_seqs > kTailMaxSeqs ||
      entries > kTailMaxUnits || tail_splits > 255 || a.done == nullptr)
    return PKV_ERR_UNSUPPORTED;
  const int smem = tail_smem_bytes(NW, NS, a.num_seqs, static_cast<int>(entries));
  constexpr int kMaxSmem = tail_smem_bytes(NW, NS, kTailMaxSeqs, kTailMaxUnits);
  static_assert(kMaxSmem <= 227 * 1024, "the largest unit list fits one CTA's shared memory");
  auto kernel = tail_stream_kernel<KV, Q, NW, NS, LEAD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaGetDevice", e);
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  // per device: the SM count, and the CTAs per SM at the last shared-memory size
  static std::atomic<int> sms_of[64];
  static std::atomic<int64_t> occ_of[64];  // (smem << 8) | CTAs per SM
  static std::atomic<uint64_t> configured{0};
  int sms = sms_of[dev].load();
  if (sms <= 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms <= 0) return cuda_fail("pkv_attention_decode: SM count", e);
    sms_of[dev].store(sms);
  }
  if (!(configured.load() & (uint64_t{1} << dev))) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: cudaFuncSetAttribute", e);
    prefer_max_shared(kernel, configured);
  }
  int per_sm = 0;
  const int64_t cached = occ_of[dev].load();
  if (cached >> 8 == smem) {
    per_sm = static_cast<int>(cached & 255);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * NW, smem);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: occupancy", e);
    occ_of[dev].store((static_cast<int64_t>(smem) << 8) | std::min(per_sm, 255));
  }
  if (per_sm <= 0) return PKV_ERR_UNSUPPORTED;
  const int64_t units = entries * a.num_kv_heads;
  const int ctas = static_cast<int>(
      std::min<int64_t>(static_cast<int64_t>(sms) * per_sm, (units + NW - 1) / NW));
  e = launch_dependent(kernel, dim3(ctas), 32 * NW, smem, st, a, kmap, vmap);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode: launch", e);
  return check_launch("pkv_attention_decode (tail queue)");
}

// Query groups of up to 8 heads take the head-columns form.  Behind a
// shared-prefix pass the contexts left are short: 16-bit head_dim-128 caches
// take a narrow form there (one warp per CTA at block size 16, two at 32:
// eleven or six CTAs per SM, so more CTAs overlap the fixed latency each
// spends reading its length, block ids and first tile and merging), when the
// partition fits its 512-entry table.
template <typename KV, typename Q, int D, int T>
pkv_status launch_dt(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     cudaStream_t st) {
  if constexpr (!std::is_same<KV, E4M3>::value && D == 128) {
    if constexpr (T == 16) {
      if (a.prefix_tokens > 0 && a.tail_queue) {
        const pkv_status s = launch_tail<KV, Q>(a, kmap, vmap, st);
        if (s != PKV_ERR_UNSUPPORTED) return s;
      }
    }
    if (a.prefix_tokens > 0 && a.group <= 8 && a.partition / T <= kMaxTableEntries2)
      return launch_form<KV, Q, D, T, true, (T == 16 ? 1 : 2)>(a, kmap, vmap, st);
  }
  return a.group <= 8 ? launch_form<KV, Q, D, T, true>(a, kmap, vmap, st)
                      : launch_form<KV, Q, D, T, false>(a, kmap, vmap, st);
}

}  // namespace tc

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
