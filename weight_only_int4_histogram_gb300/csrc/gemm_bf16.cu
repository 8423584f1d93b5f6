// BF16-activation instantiations of the grouped W4A16 GEMM.
#include "gemm.cuh"

namespace w4a16 {
template cudaError_t launch_gemm_dt<DT_BF16>(int, int, const GemmParams&, const CUtensorMap&,
                                              const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                              int, int, cudaStream_t, bool);
}
