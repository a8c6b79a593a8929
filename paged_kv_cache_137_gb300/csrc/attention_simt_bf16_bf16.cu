// CUDA-core decode attention kernels for a BF16 cache with BF16 queries.
#include "attention_simt.cuh"

namespace pkv {
template pkv_status launch_decode_simt<BF16, BF16>(const DecodeArgs&, int, int, cudaStream_t);
}  // namespace pkv
