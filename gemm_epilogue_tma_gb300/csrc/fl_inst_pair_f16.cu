// CTA-pair kernel instances (f16): 256 x 128 and 256 x 256 tiles on two SMs,
// and 256 x 256 tiles split over K between two pairs.
#include "fl_pair_kernel.cuh"

namespace fl {
template cudaError_t launch_pair<DT_F16, 128, PRO_NONE, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_NONE, 1>();
template cudaError_t launch_pair<DT_F16, 128, PRO_RMS, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_RMS, 1>();
template cudaError_t launch_pair<DT_F16, 128, PRO_LN, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_LN, 1>();
template cudaError_t launch_pair<DT_F16, 256, PRO_NONE, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_NONE, 1>();
template cudaError_t launch_pair<DT_F16, 256, PRO_RMS, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_RMS, 1>();
template cudaError_t launch_pair<DT_F16, 256, PRO_LN, 1>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_LN, 1>();
template cudaError_t launch_pair<DT_F16, 256, PRO_NONE, 2>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_NONE, 2>();
template cudaError_t launch_pair<DT_F16, 256, PRO_RMS, 2>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_RMS, 2>();
template cudaError_t launch_pair<DT_F16, 256, PRO_LN, 2>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_LN, 2>();
}  // namespace fl
