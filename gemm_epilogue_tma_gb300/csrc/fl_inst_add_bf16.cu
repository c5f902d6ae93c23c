// Instances with the input-bias prologue (A + b along K) (bf16): the tile,
// CTA-pair and split-K kernels.
#include "fl_gemm_kernel.cuh"
#include "fl_pair_kernel.cuh"
#include "fl_splitk_kernel.cuh"

namespace fl {
template cudaError_t launch_gemm<DT_BF16, 128, PRO_ADD, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<DT_BF16, 256, PRO_ADD, false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_pair<DT_BF16, 128, PRO_ADD, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 128, PRO_ADD, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_ADD, 1, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_ADD, 1>();
template cudaError_t launch_pair<DT_BF16, 256, PRO_ADD, 2, false>(const GemmParams&, int, cudaStream_t);
template int pair_max_clusters<DT_BF16, 256, PRO_ADD, 2>();
template cudaError_t launch_splitk<DT_BF16, 64, PRO_ADD>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_splitk<DT_BF16, 128, PRO_ADD>(const GemmParams&, int, int, cudaStream_t);
template int splitk_max_clusters<DT_BF16, 64, PRO_ADD>(int, int);
template int splitk_max_clusters<DT_BF16, 128, PRO_ADD>(int, int);
}  // namespace fl
