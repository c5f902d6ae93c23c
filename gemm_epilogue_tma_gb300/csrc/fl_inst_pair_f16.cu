// CTA-pair kernel instances (f16): 256 x 128 and 256 x 256 tiles on two SMs.
#include "fl_pair_kernel.cuh"

namespace fl {
template cudaError_t launch_pair<DT_F16, 128, PRO_NONE>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_NONE>();
template cudaError_t launch_pair<DT_F16, 128, PRO_RMS>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_RMS>();
template cudaError_t launch_pair<DT_F16, 128, PRO_LN>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 128, PRO_LN>();
template cudaError_t launch_pair<DT_F16, 256, PRO_NONE>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_NONE>();
template cudaError_t launch_pair<DT_F16, 256, PRO_RMS>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_RMS>();
template cudaError_t launch_pair<DT_F16, 256, PRO_LN>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_F16, 256, PRO_LN>();
}  // namespace fl
