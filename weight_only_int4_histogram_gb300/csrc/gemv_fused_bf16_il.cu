// BF16-activation instantiations of the fused CUDA-core expert GEMMs, relaid-out (interleaved) weights.
#include "gemv_fused.cuh"

namespace w4a16 {
template cudaError_t launch_gemv_fused_dt<DT_BF16, LAYOUT_IL>(int, const FusedParams&, const CUtensorMap&,
                                                         const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                         int, int, cudaStream_t, bool);
}
