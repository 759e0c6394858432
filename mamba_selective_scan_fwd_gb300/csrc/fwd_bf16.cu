// Forward kernels for bf16 io (one translation unit per io type, compiled in parallel).
#include "fwd.cuh"

namespace ss {
template cudaError_t launch_fwd_io<__nv_bfloat16>(const FwdArgs&, const FPlan&, cudaStream_t, int, float*,
                                              const TmaMaps&);
}  // namespace ss
