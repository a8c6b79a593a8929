// CUDA-core decode attention kernels for a E4M3 cache with F16 queries.
#include "attention_simt.cuh"

namespace pkv {
template pkv_status launch_decode_simt<E4M3, F16>(const DecodeArgs&, int, int, cudaStream_t);
}  // namespace pkv
