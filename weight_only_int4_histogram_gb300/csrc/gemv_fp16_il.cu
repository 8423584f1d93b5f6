// FP16-activation instantiations of the grouped W4A16 GEMV (CUDA cores), relaid-out (interleaved) weights.
#include "gemv.cuh"

namespace w4a16 {
template cudaError_t launch_gemv_dt<DT_FP16, LAYOUT_IL>(int, int, const GemmParams&, const CUtensorMap&,
                                                     const CUtensorMap&, int, int, cudaStream_t, bool);
}
