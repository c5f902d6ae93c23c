// Multi-output instances (bf16): one RMSNorm / LayerNorm activation feeding
// several weights, on the CTA-pair, split-K and tile kernels.
#include "fl_gemm_kernel.cuh"
#include "fl_pair_kernel.cuh"
#include "fl_splitk_kernel.cuh"

namespace fl {
template cudaError_t launch_pair<DT_BF16, 256, PRO_RMS, 1, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_pair<DT_BF16, 256, PRO_LN, 1, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_pair<DT_BF16, 256, PRO_RMS, 2, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_pair<DT_BF16, 256, PRO_LN, 2, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 64, PRO_RMS, false, true>(const GemmParamsMulti&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 64, PRO_LN, false, true>(const GemmParamsMulti&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_RMS, false, true>(const GemmParamsMulti&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_LN, false, true>(const GemmParamsMulti&, int, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 128, PRO_RMS, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 256, PRO_RMS, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 128, PRO_LN, false, true>(const GemmParamsMulti&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 256, PRO_LN, false, true>(const GemmParamsMulti&, int, cudaStream_t);
}  // namespace fl
