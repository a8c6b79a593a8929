// Tensor-core decode attention kernel for a F16 cache with F16 queries.
#include "attention_tc_launch.cuh"

namespace pkv {
template pkv_status launch_decode_tc<F16, F16>(const DecodeArgs&, int, const CUtensorMap&,
                                              const CUtensorMap&, cudaStream_t);
}  // namespace pkv
