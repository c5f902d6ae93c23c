// Tile-kernel instances without a prologue (f16): the seven GEMM-first
// patterns and the FFN down projection.
#include "fl_gemm_kernel.cuh"

namespace fl {
template cudaError_t launch_gemm<DT_F16, 128, PRO_NONE, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_F16, 256, PRO_NONE, false>(const GemmParams&, int, cudaStream_t);
}  // namespace fl
