// Tile-kernel instances with a norm prologue (bf16): RMSNorm / LayerNorm GEMM
// and the SwiGLU gate/up kernel.
#include "fl_gemm_kernel.cuh"

namespace fl {
template cudaError_t launch_gemm<DT_BF16, 128, PRO_RMS, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 256, PRO_RMS, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 128, PRO_LN, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 256, PRO_LN, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 128, PRO_RMS, true>(const GemmParams&, int, cudaStream_t);
}  // namespace fl
