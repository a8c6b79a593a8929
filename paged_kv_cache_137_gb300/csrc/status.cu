// The library's device error word and the stage-wait limit.
//
// Inputs that only the GPU reads (block-table entries, context lengths, a
// declared shared prefix) cannot be checked on the host without a copy, and a
// bounded wait that gives up happens on the GPU as well.  The attention
// kernels turn the affected outputs into NaN and OR a PKV_DEVICE_* bit into
// one int per device, declared here as a file-scope device variable.  Its
// name in host code is only a host-side stand-in, so the host asks the
// runtime for its device address (cudaGetSymbolAddress, once per device,
// with that device current) and passes that address to the kernels.
#include <atomic>
#include <mutex>

#include "attention.h"
#include "device_common.cuh"

namespace pkv {
namespace {

static __device__ __align__(16) int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
std::atomic<int*> g_addr[kMaxDevices];
std::atomic<uint64_t> g_wait_ns{50000000ull};

}  // namespace

int* device_status_word(pkv_status* st) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail("device error word: cudaGetDevice", e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = fail(PKV_ERR_UNSUPPORTED, "device index above 63");
    return nullptr;
  }
  int* p = g_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_mu);
  p = g_addr[dev].load(std::memory_order_relaxed);
  if (!p) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_device_status);
    if (e != cudaSuccess || a == nullptr) {
      *st = e != cudaSuccess ? cuda_fail("device error word: cudaGetSymbolAddress", e)
                             : fail(PKV_ERR_CUDA, "device error word: no address");
      return nullptr;
    }
    p = static_cast<int*>(a);
    g_addr[dev].store(p, std::memory_order_release);
  }
  return p;
}

uint64_t stage_wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_device_status(int32_t* flags, int32_t clear, void* stream) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  pkv_status st = PKV_OK;
  int* word = device_status_word(&st);
  if (!word) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("pkv_device_status: reading the error word", e);
  if (clear) {
    e = cudaMemsetAsync(word, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail("pkv_device_status: clearing the error word", e);
  }
  *flags = v;
  return PKV_OK;
}

extern "C" pkv_status pkv_set_stage_wait_limit(uint64_t nanoseconds) {
  g_wait_ns.store(nanoseconds, std::memory_order_relaxed);
  return PKV_OK;
}
