// CTA-pair kernel instances (bf16): 256 x 128 and 256 x 256 tiles on two SMs,
// 256 x 256 tiles split over K between two pairs, and the SwiGLU gate/up
// pair (RMS prologue, Wg and Wu stacked in one 256-row weight tile).
#include "fl_pair_kernel.cuh"

namespace fl {
template cudaError_t launch_pair<DT_BF16, 128, PRO_NONE, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 128, PRO_NONE, 1>();
template cudaError_t launch_pair<DT_BF16, 128, PRO_RMS, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 128, PRO_RMS, 1>();
template cudaError_t launch_pair<DT_BF16, 128, PRO_LN, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 128, PRO_LN, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_NONE, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_NONE, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_RMS, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_RMS, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_LN, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_LN, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_NONE, 2, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_NONE, 2>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_RMS, 2, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_RMS, 2>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_LN, 2, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_LN, 2>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_RMS, 1, true>(const GemmParams&, int, cudaStream_t);
}  // namespace fl
