// Backward kernels for bf16 io (one translation unit per io type, compiled in parallel).
#include "bwd2.cuh"

namespace ss {
template cudaError_t launch_bwd2_io<__nv_bfloat16>(const BwdArgs&, const FPlan&, cudaStream_t, float*);
}  // namespace ss
