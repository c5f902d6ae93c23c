// Standalone RMSNorm: y = x * gamma / sqrt(mean_k(x^2) + eps), rounded once to
// the dtype. For a normalised activation that several consumers read (the
// case where folding the norm into each consumer's GEMM would recompute it),
// written after the generated RMSNorm kernel of the "hackable compiler" post
// (sum of squares, times 1/K, plus eps, rsqrt, times x, times the weight).
//
// Bound by HBM: x is read once and y written once. One warp per row (rows
// grid-stride over at most two CTAs per SM, so no partial last wave); every
// lane moves 16-byte vectors at a 512-byte stride (coalesced across the
// warp). Rows of up to 4096 elements stay in registers between the sum of
// squares and the scaling (16 vectors per lane, all issued before the first
// is used), and gamma is staged once per CTA in shared memory; longer rows
// are read a second time, from L2, for the scaling.
// The lanes' partial sums are added by a fixed butterfly, so the result does
// not depend on timing. y may be x itself: every element is read before the
// thread that reads it writes it, and the sum is complete before any write.
#include "fl_common.cuh"
#include "fl_internal.h"

namespace fl {

namespace {

constexpr int kVecPerLane = 16;  // register-resident row: 16 x 8 elements per lane, 4096 per warp

template <int DT>
__device__ __forceinline__ void sq_acc_vec(const uint4& v, float& s0, float& s1) {
    using Ops = DTypeOps<DT>;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = Ops::unpack(w[e]);
        s0 = fmaf(f.x, f.x, s0);
        s1 = fmaf(f.y, f.y, s1);
    }
}

template <int DT>
__device__ __forceinline__ uint4 scale_vec(const uint4& v, const uint4& g, float r) {
    using Ops = DTypeOps<DT>;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = Ops::unpack(w[e]), gg = Ops::unpack(gw[e]);
        o[e] = Ops::pack(f.x * r * gg.x, f.y * r * gg.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One row longer than 4096 elements, by one warp.
template <int DT>
__device__ __forceinline__ void rms_norm_row(const uint16_t* x, const uint16_t* __restrict__ gamma, uint16_t* y,
                                             int row, int K, float eps, int lane);

template <int DT>
__global__ void __launch_bounds__(256, 2) fl_rms_norm_kernel(const uint16_t* x, const uint16_t* __restrict__ gamma,
                                                             uint16_t* y, int M, int K, float eps) {
    griddep_wait();  // x may come from the previous kernel on the stream
    const int lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (K <= 256 * kVecPerLane) {
        // gamma is the same for every row: staged once per CTA in shared
        // memory (one memory round trip per row instead of two)
        __shared__ uint4 gs[256 * kVecPerLane / 8];
        for (int i = threadIdx.x; i < K / 8; i += blockDim.x) gs[i] = ldg_v4(gamma + i * 8);
        __syncthreads();
        for (int row = row0; row < M; row += gridDim.x * 8) {
            const uint16_t* xr = x + (size_t)row * K;
            uint16_t* yr = y + (size_t)row * K;
            uint4 v[kVecPerLane];
#pragma unroll
            for (int u = 0; u < kVecPerLane; ++u)
                if (lane * 8 + u * 256 < K) v[u] = ldg_v4(xr + lane * 8 + u * 256);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int u = 0; u < kVecPerLane; ++u)
                if (lane * 8 + u * 256 < K) sq_acc_vec<DT>(v[u], s0, s1);
            const float r = rsqrtf(warp_sum(s0 + s1) / (float)K + eps);
#pragma unroll
            for (int u = 0; u < kVecPerLane; ++u) {
                const int k = lane * 8 + u * 256;
                if (k < K) *reinterpret_cast<uint4*>(yr + k) = scale_vec<DT>(v[u], gs[k / 8], r);
            }
        }
    } else {
        for (int row = row0; row < M; row += gridDim.x * 8) rms_norm_row<DT>(x, gamma, y, row, K, eps, lane);
    }
    // The next kernel is let in only once this CTA's rows are done: letting
    // it in earlier would park its CTAs on SM slots this grid still needs.
    griddep_launch_dependents();
}

template <int DT>
__device__ __forceinline__ void rms_norm_row(const uint16_t* x, const uint16_t* __restrict__ gamma, uint16_t* y,
                                             int row, int K, float eps, int lane) {
    const uint16_t* xr = x + (size_t)row * K;
    uint16_t* yr = y + (size_t)row * K;
    float s0 = 0.f, s1 = 0.f;
    // long rows: sum of squares, then a second read for the scaling
    for (int k0 = lane * 8; k0 < K; k0 += 256 * 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (k0 + u * 256 < K) v[u] = ldg_v4(xr + k0 + u * 256);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (k0 + u * 256 < K) sq_acc_vec<DT>(v[u], s0, s1);
    }
    const float r = rsqrtf(warp_sum(s0 + s1) / (float)K + eps);
    for (int k = lane * 8; k < K; k += 256)
        *reinterpret_cast<uint4*>(yr + k) = scale_vec<DT>(ldg_v4(xr + k), ldg_v4(gamma + k), r);
}

}  // namespace

cudaError_t launch_rms_norm(int dt, const void* x, const void* gamma, void* y, int M, int K, float eps, int pdl,
                            int sms, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    const int ctas = (M + 7) / 8;
    cfg.gridDim = dim3((unsigned)(ctas < 2 * sms ? ctas : 2 * sms), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint16_t* xp = static_cast<const uint16_t*>(x);
    const uint16_t* gp = static_cast<const uint16_t*>(gamma);
    uint16_t* yp = static_cast<uint16_t*>(y);
    if (dt == DT_F16) return cudaLaunchKernelEx(&cfg, fl_rms_norm_kernel<DT_F16>, xp, gp, yp, M, K, eps);
    return cudaLaunchKernelEx(&cfg, fl_rms_norm_kernel<DT_BF16>, xp, gp, yp, M, K, eps);
}

}  // namespace fl
