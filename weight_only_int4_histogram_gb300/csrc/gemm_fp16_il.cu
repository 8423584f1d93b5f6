// FP16-activation instantiations of the grouped W4A16 GEMM, relaid-out (interleaved) weights.
#include "gemm.cuh"

namespace w4a16 {
template cudaError_t launch_gemm_dt<DT_FP16, LAYOUT_IL>(int, int, const GemmParams&, const CUtensorMap&,
                                                     const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     int, int, cudaStream_t, bool);
}
