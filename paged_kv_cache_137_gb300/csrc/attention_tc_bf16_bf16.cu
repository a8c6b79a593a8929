// Tensor-core decode attention kernel for a BF16 cache with BF16 queries.
#include "attention_tc_launch.cuh"

namespace pkv {
template pkv_status launch_decode_tc<BF16, BF16>(const DecodeArgs&, int, const CUtensorMap&,
                                              const CUtensorMap&, cudaStream_t);
}  // namespace pkv
