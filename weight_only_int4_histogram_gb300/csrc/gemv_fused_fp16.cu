// FP16-activation instantiations of the fused CUDA-core expert GEMMs, checkpoint-layout weights.
#include "gemv_fused.cuh"

namespace w4a16 {
template cudaError_t launch_gemv_fused_dt<DT_FP16, LAYOUT_CANON>(int, const FusedParams&, const CUtensorMap&,
                                                         const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                         int, int, cudaStream_t, bool);
}
