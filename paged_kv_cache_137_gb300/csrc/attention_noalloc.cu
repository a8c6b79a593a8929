// Decode attention for callers that cannot allocate device memory.
//
// pkv_attention_decode keeps its split-K partial results in a workspace the
// caller allocates.  Some callers cannot do that: a plug-in hosted by another
// runtime that owns all device memory and hands the plug-in nothing but its
// input and output buffers, or a serving loop that must never call cudaMalloc
// while it runs because the call can synchronise the whole device and stall
// every stream.  pkv_attention_decode_noalloc serves them: its scratch is a
// fixed-size array in device global memory that this file declares, so the
// call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
// routine).  The array holds kNoAllocScratchBytes on every GPU that loads the
// library, until the process exits.
//
// The host needs the array's device address: the array's name in host code
// is only a host-side stand-in, and a kernel handed that stand-in would fault
// or, where the GPU can reach host memory, silently use the wrong memory.  The
// first call on a device (with that device current) asks the runtime for the
// address with cudaGetSymbolAddress and caches it per device; that first call
// should come before any stream capture.
//
// Every call on a device shares the one array, which keeps whatever the last
// call left in it.  Only the split-K arrival counters at its start must be
// zero when a call begins.  A call that runs to completion leaves them zero
// (the CTA that merges a sequence's splits resets its counter, also after a
// wait gave up); each call still clears them on its stream before the
// decode kernel runs (a memset, not an allocation), so that a call that never
// completed (its process or context torn down mid-kernel) cannot leave a
// count behind for the next one.  Every other scratch value is written before
// it is read within the same call.  Calls that overlap on the GPU (two
// streams at once) race on the array.  The array's address is looked up once
// per device and kept: cudaDeviceReset while the library is loaded is not
// supported.
#include <mutex>

#include "attention.h"
#include "device_common.cuh"

namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
pkv_status scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("pkv_attention_decode_noalloc: cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return fail(PKV_ERR_UNSUPPORTED, "pkv_attention_decode_noalloc: device index above 63");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode_noalloc: cudaGetSymbolAddress", e);
    if (p == nullptr)
      return fail(PKV_ERR_CUDA, "pkv_attention_decode_noalloc: cudaGetSymbolAddress gave NULL");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_attention_decode_noalloc(
    void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, const pkv_kv_desc* desc, float softmax_scale,
    float k_scale, float v_scale, int32_t partition_tokens, void* stream) {
  const size_t need = pkv_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc,
                                                    partition_tokens);
  if (need > kNoAllocScratchBytes) {
    set_error("pkv_attention_decode_noalloc: these sizes need %zu bytes of split-K scratch, "
              "more than the fixed %zu; use pkv_attention_decode with a workspace or a larger "
              "partition_tokens",
              need, kNoAllocScratchBytes);
    return PKV_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  if (need > 0) {
    const pkv_status st = scratch_on_current_device(&scratch);
    if (st != PKV_OK) return st;
    const size_t counters = attention_counter_bytes(num_seqs, num_q_heads, max_blocks, desc,
                                                    partition_tokens);
    const cudaError_t e = cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("pkv_attention_decode_noalloc: clearing the counters", e);
  }
  return pkv_attention_decode(out, q, q_dtype, k_cache, v_cache, block_tables, max_blocks,
                              context_lens, num_seqs, num_q_heads, desc, softmax_scale, k_scale,
                              v_scale, partition_tokens, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                              stream);
}
