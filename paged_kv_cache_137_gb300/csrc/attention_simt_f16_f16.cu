// CUDA-core decode attention kernels for a F16 cache with F16 queries.
#include "attention_simt.cuh"

namespace pkv {
template pkv_status launch_decode_simt<F16, F16>(const DecodeArgs&, int, int, cudaStream_t);
}  // namespace pkv
