// Backward kernels for f32 io (one translation unit per io type, compiled in parallel).
#include "bwd.cuh"

namespace ss {
template cudaError_t launch_bwd_io<float>(const BwdArgs&, const FPlan&, cudaStream_t, float*, const TmaMaps&,
                                              const TmaMaps&);
}  // namespace ss
