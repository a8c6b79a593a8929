// CUDA-core decode attention kernels for a F32 cache with F32 queries.
#include "attention_simt.cuh"

namespace pkv {
template pkv_status launch_decode_simt<F32, F32>(const DecodeArgs&, int, int, cudaStream_t);
}  // namespace pkv
