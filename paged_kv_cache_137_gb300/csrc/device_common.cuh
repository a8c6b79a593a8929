// Device helpers shared by the libpkv kernels: element loads converted to
// fp32, E4M3 conversions through the hardware cvt instructions, and host
// launch-error mapping.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "common.h"

namespace pkv {

// Storage tags: the element type a cache or an input holds.
struct F32 { using raw = float; static constexpr int bytes = 4; };
struct F16 { using raw = __half; static constexpr int bytes = 2; };
struct BF16 { using raw = __nv_bfloat16; static constexpr int bytes = 2; };
struct E4M3 { using raw = uint8_t; static constexpr int bytes = 1; };

// ---------------------------------------------------------------- E4M3 cvt
// Two E4M3 bytes (low byte = first element) -> two f16 values, exact.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return *reinterpret_cast<__half2*>(&r);
}

// Two fp32 values -> two E4M3 bytes (first in the low byte), round to
// nearest even, finite overflow saturated to +/-448, NaN kept.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float first, float second) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

// ------------------------------------------------------- loads as fp32
// Load N consecutive elements (N * bytes must be 4, 8 or 16 bytes, and the
// address aligned to that size) and convert them to fp32.
template <typename Tag, int N>
struct LoadF32;

template <int N>
struct LoadF32<F32, N> {
  static __device__ __forceinline__ void run(const void* p, float* f) {
    static_assert(N == 1 || N == 2 || N == 4 || N == 8, "");
    if constexpr (N == 8) {
      const float4 a = reinterpret_cast<const float4*>(p)[0];
      const float4 b = reinterpret_cast<const float4*>(p)[1];
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
      f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else if constexpr (N == 4) {
      const float4 a = *reinterpret_cast<const float4*>(p);
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    } else if constexpr (N == 2) {
      const float2 a = *reinterpret_cast<const float2*>(p);
      f[0] = a.x; f[1] = a.y;
    } else {
      f[0] = *reinterpret_cast<const float*>(p);
    }
  }
};

template <typename W>
__device__ __forceinline__ void unpack_bf16(const W& w, float* f, int n) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
  for (int i = 0; i < n / 2; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

template <typename W>
__device__ __forceinline__ void unpack_f16(const W& w, float* f, int n) {
  const __half2* h = reinterpret_cast<const __half2*>(&w);
  for (int i = 0; i < n / 2; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

template <typename W>
__device__ __forceinline__ void unpack_e4m3(const W& w, float* f, int n) {
  const uint16_t* u = reinterpret_cast<const uint16_t*>(&w);
  for (int i = 0; i < n / 2; ++i) {
    const float2 x = __half22float2(e4m3x2_to_half2(u[i]));
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

template <int BYTES>
struct Word;
template <> struct Word<2> { using type = uint16_t; };
template <> struct Word<4> { using type = uint32_t; };
template <> struct Word<8> { using type = uint2; };
template <> struct Word<16> { using type = uint4; };

template <int N>
struct LoadF32<BF16, N> {
  static __device__ __forceinline__ void run(const void* p, float* f) {
    using W = typename Word<2 * N>::type;
    const W w = *reinterpret_cast<const W*>(p);
    unpack_bf16(w, f, N);
  }
};

template <int N>
struct LoadF32<F16, N> {
  static __device__ __forceinline__ void run(const void* p, float* f) {
    using W = typename Word<2 * N>::type;
    const W w = *reinterpret_cast<const W*>(p);
    unpack_f16(w, f, N);
  }
};

template <int N>
struct LoadF32<E4M3, N> {
  static __device__ __forceinline__ void run(const void* p, float* f) {
    using W = typename Word<N>::type;
    const W w = *reinterpret_cast<const W*>(p);
    unpack_e4m3(w, f, N);
  }
};

// Store one fp32 value as the element type of an output (round to nearest).
template <typename Tag>
__device__ __forceinline__ void store_elem(void* base, size_t idx, float x);
template <> __device__ __forceinline__ void store_elem<F32>(void* b, size_t i, float x) {
  static_cast<float*>(b)[i] = x;
}
template <> __device__ __forceinline__ void store_elem<F16>(void* b, size_t i, float x) {
  static_cast<__half*>(b)[i] = __float2half_rn(x);
}
template <> __device__ __forceinline__ void store_elem<BF16>(void* b, size_t i, float x) {
  static_cast<__nv_bfloat16*>(b)[i] = __float2bfloat16_rn(x);
}

template <typename Tag>
__device__ __forceinline__ float load_elem(const void* b, size_t i);
template <> __device__ __forceinline__ float load_elem<F32>(const void* b, size_t i) {
  return static_cast<const float*>(b)[i];
}
template <> __device__ __forceinline__ float load_elem<F16>(const void* b, size_t i) {
  return __half2float(static_cast<const __half*>(b)[i]);
}
template <> __device__ __forceinline__ float load_elem<BF16>(const void* b, size_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(b)[i]);
}

// ------------------------------------------------------------ host side
// Ask once per device for the largest shared-memory carveout for `kernel` (a
// hint the driver may follow).  The attention kernels run with it; a small
// kernel launched between them that asks for the same split spares the SMs a
// reconfiguration of their shared memory and L1.  Failures are cleared and
// ignored (the kernel then runs with the driver's choice).
template <typename Kernel>
inline void prefer_max_shared(Kernel kernel, std::atomic<uint64_t>& configured) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return;
  }
  const uint64_t bit = uint64_t{1} << dev;
  if (configured.load() & bit) return;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    (void)cudaGetLastError();
  configured.fetch_or(bit);
}

inline pkv_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// A failed runtime call: record the message and clear the runtime's sticky
// last-error slot so that a later launch check does not report it again.
inline pkv_status cuda_fail(const char* what, cudaError_t e) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  (void)cudaGetLastError();
  return PKV_ERR_CUDA;
}

// Store 8 consecutive K/V elements of the source type into the cache type:
// a plain copy for a 16/32-bit cache (which stores the input type), or
// x * inv rounded to E4M3 (nearest even, saturating) for an E4M3 cache.
// src and dst are 8-element aligned.
template <typename Src, typename Dst>
__device__ __forceinline__ void store8(const void* src, void* dst, float inv) {
  if constexpr (std::is_same<Dst, E4M3>::value) {
    float f[8];
    LoadF32<Src, 8>::run(src, f);
    uint2 packed;
    uint16_t* q = reinterpret_cast<uint16_t*>(&packed);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = f32x2_to_e4m3x2(f[2 * i] * inv, f[2 * i + 1] * inv);
    *reinterpret_cast<uint2*>(dst) = packed;
  } else {
    static_assert(std::is_same<Src, Dst>::value, "16/32-bit caches store the input type");
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < Src::bytes / 2; ++i) d[i] = s[i];
  }
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline pkv_status check_desc(const pkv_kv_desc* d) {
  if (!d) return fail(PKV_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "desc sizes must be positive");
  if (d->kv_dtype < PKV_F32 || d->kv_dtype > PKV_E4M3)
    return fail(PKV_ERR_INVALID_ARG, "unknown kv_dtype");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (d->block_size != 16 && d->block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "block_size must be 16 or 32");
  if (d->head_scales != nullptr) {
    if (d->kv_dtype != PKV_E4M3) return fail(PKV_ERR_INVALID_ARG, "head_scales need an E4M3 cache");
    if (!aligned(d->head_scales, 4)) return fail(PKV_ERR_INVALID_ARG, "head_scales misaligned");
  }
  return PKV_OK;
}

// Scales of KV head h of an E4M3 cache: the per-head table when there is one
// ([4][n_kv]: K scale, V scale, K inverse, V inverse), else the per-tensor
// values.  qk folds the K scale into the log2-domain logit scale in the
// order the host folds a per-tensor one: (softmax_scale * k_scale) * log2(e).
struct HeadScales {
  float qk, v, k_inv, v_inv;
};
__device__ __forceinline__ HeadScales head_scales(const float* table, int n_kv, int h,
                                                  float softmax_scale, float qk, float v,
                                                  float k_inv, float v_inv) {
  if (table == nullptr) return {qk, v, k_inv, v_inv};
  return {(softmax_scale * table[h]) * 1.4426950408889634f, table[n_kv + h], table[2 * n_kv + h],
          table[3 * n_kv + h]};
}

}  // namespace pkv
