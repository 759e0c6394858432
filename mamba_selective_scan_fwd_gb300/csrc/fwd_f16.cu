// Forward kernels for f16 io (one translation unit per io type, compiled in parallel).
#include "fwd.cuh"

namespace ss {
template cudaError_t launch_fwd_io<__half>(const FwdArgs&, const FPlan&, cudaStream_t, int, float*,
                                              const TmaMaps&);
}  // namespace ss
