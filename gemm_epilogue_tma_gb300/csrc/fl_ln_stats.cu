// LayerNorm row statistics: mean and 1/sqrt(var + eps) of every activation row,
// computed once per call ahead of the fused GEMM kernels, which fold
// (x - mean) * rstd * gamma + beta into their staged operand. Only these 8
// bytes per row go through memory; the normalised activation never does.
//
// One warp per row: every lane reads 16-byte vectors at a 512-byte stride
// (coalesced across the warp), all issued before any is used, and
// accumulates sums shifted by the mean of the row's first eight elements,
// S1 = sum(x - c) and S2 = sum((x - c)^2), which keeps the variance free of
// cancellation for rows far from zero. A fixed butterfly adds the lanes'
// sums, so results do not depend on timing.
#include "fl_common.cuh"
#include "fl_internal.h"

namespace fl {

template <int DT>
__global__ void __launch_bounds__(256) fl_ln_stats_kernel(const uint16_t* __restrict__ x, int M, int K, float eps,
                                                           float2* __restrict__ stats) {
    using Ops = DTypeOps<DT>;
    // x may come from the previous kernel on the stream
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= M) return;
    const uint16_t* xr = x + (size_t)row * K;
    // Up to 16 vectors per lane in flight (a 4096-wide row in one round trip);
    // the shift comes with them.
    constexpr int U = 16;
    const uint4 h = ldg_v4(xr);
    float s1[2] = {0.f, 0.f}, s2[2] = {0.f, 0.f};
    float c = 0.f;
#pragma unroll 1
    for (int k0 = lane * 8; k0 < K; k0 += U * 256) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (k0 + u * 256 < K) v[u] = ldg_v4(xr + k0 + u * 256);
        if (k0 == lane * 8) {
            const float2 a = Ops::unpack(h.x), b = Ops::unpack(h.y), d = Ops::unpack(h.z), e = Ops::unpack(h.w);
            c = (((a.x + a.y) + (b.x + b.y)) + ((d.x + d.y) + (e.x + e.y))) * 0.125f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u * 256 < K) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Ops::unpack(w[e]);
                    const float d0 = f.x - c, d1 = f.y - c;
                    s1[u & 1] += d0 + d1;
                    s2[u & 1] = fmaf(d0, d0, fmaf(d1, d1, s2[u & 1]));
                }
            }
        }
    }
    float a1 = s1[0] + s1[1], a2 = s2[0] + s2[1];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
        a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    }
    if (lane == 0) {
        const float inv_k = 1.0f / (float)K;
        const float d = a1 * inv_k;  // mean - c
        const float var = fmaxf(fmaf(-d, d, a2 * inv_k), 0.f);
        stats[row] = make_float2(c + d, rsqrtf(var + eps));
    }
}

cudaError_t launch_ln_stats(int dt, const void* x, int M, int K, float eps, void* stats, int pdl,
                            cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + 7) / 8), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint16_t* xp = static_cast<const uint16_t*>(x);
    float2* sp = static_cast<float2*>(stats);
    if (dt == DT_F16) return cudaLaunchKernelEx(&cfg, fl_ln_stats_kernel<DT_F16>, xp, M, K, eps, sp);
    return cudaLaunchKernelEx(&cfg, fl_ln_stats_kernel<DT_BF16>, xp, M, K, eps, sp);
}

}  // namespace fl
