// Split-K kernel instances (bf16): few output tiles, weights streamed once; the
// SwiGLU gate/up form (two weights) for decode row counts.
#include "fl_splitk_kernel.cuh"

namespace fl {
template cudaError_t launch_splitk<DT_BF16, 64, PRO_NONE>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 64, PRO_RMS>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 64, PRO_LN>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_NONE>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_RMS>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_LN>(const GemmParams&, int, int, cudaStream_t);
template int splitk_max_clusters<DT_BF16, 64, PRO_NONE>(int, int);
template int splitk_max_clusters<DT_BF16, 64, PRO_RMS>(int, int);
template int splitk_max_clusters<DT_BF16, 64, PRO_LN>(int, int);
template int splitk_max_clusters<DT_BF16, 128, PRO_NONE>(int, int);
template int splitk_max_clusters<DT_BF16, 128, PRO_RMS>(int, int);
template int splitk_max_clusters<DT_BF16, 128, PRO_LN>(int, int);
template cudaError_t launch_splitk<DT_BF16, 64, PRO_RMS, true>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_RMS, true>(const GemmParams&, int, int, cudaStream_t);
template int splitk_max_clusters<DT_BF16, 64, PRO_RMS, true>(int, int);
template int splitk_max_clusters<DT_BF16, 128, PRO_RMS, true>(int, int);
}  // namespace fl
