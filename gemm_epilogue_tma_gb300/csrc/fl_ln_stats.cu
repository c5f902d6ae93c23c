// LayerNorm row statistics: mean and 1/sqrt(var + eps) of every activation row,
// computed once per call ahead of the fused GEMM kernels, which fold
// (x - mean) * rstd * gamma + beta into their staged operand. Only these 8
// bytes per row go through memory; the normalised activation never does.
//
// Persistent warps take the rows grid-stride, each row in halves of 2048
// elements (8 16-byte vectors per lane, coalesced across the warp), double
// buffered: the next half's loads (of this row or the warp's next row) are in
// flight while this half is summed, so a warp never waits for a whole row's
// round trip between rows. Sums are shifted by the mean of the row's first
// eight elements, S1 = sum(x - c) and S2 = sum((x - c)^2), which keeps the
// variance free of cancellation for rows far from zero. A fixed butterfly
// adds the lanes' sums, so results do not depend on timing.
#include "fl_common.cuh"
#include "fl_internal.h"

namespace fl {

namespace {

constexpr int kHalfVec = 8;                      // vectors per lane per half row
constexpr int kHalfElems = 32 * kHalfVec * 8;    // 2048 elements

__device__ __forceinline__ void load_half(uint4 (&buf)[kHalfVec], const uint16_t* x, int row, int h, int K,
                                          int lane) {
#pragma unroll
    for (int u = 0; u < kHalfVec; ++u) {
        const int k = h * kHalfElems + lane * 8 + u * 256;
        buf[u] = k < K ? ldg_v4(x + (size_t)row * K + k) : make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(256, 2) fl_ln_stats_kernel(const uint16_t* __restrict__ x, int M, int K, float eps,
                                                              float2* __restrict__ stats) {
    using Ops = DTypeOps<DT>;
    // x may come from the previous kernel on the stream
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * 8;
    const int nh = (K + kHalfElems - 1) / kHalfElems;
    int row = blockIdx.x * 8 + (threadIdx.x >> 5), h = 0, q = 0;
    uint4 A[kHalfVec], B[kHalfVec];
    if (row < M) load_half(A, x, row, 0, K, lane);
    float s1 = 0.f, s2 = 0.f, c = 0.f;
    auto sum_half = [&](const uint4 (&buf)[kHalfVec]) {
        if (h == 0) {
            // the shift: mean of the row's first eight elements (lane 0's first vector)
            const float2 a = Ops::unpack(buf[0].x), b = Ops::unpack(buf[0].y), d = Ops::unpack(buf[0].z),
                         e = Ops::unpack(buf[0].w);
            c = __shfl_sync(0xffffffffu, (((a.x + a.y) + (b.x + b.y)) + ((d.x + d.y) + (e.x + e.y))) * 0.125f, 0);
            s1 = s2 = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kHalfVec; ++u) {
            if (h * kHalfElems + lane * 8 + u * 256 < K) {
                const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Ops::unpack(w[e]);
                    const float d0 = f.x - c, d1 = f.y - c;
                    s1 += d0 + d1;
                    s2 = fmaf(d0, d0, fmaf(d1, d1, s2));
                }
            }
        }
        if (h == nh - 1) {
            float a1 = s1, a2 = s2;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a1 += __shfl_xor_sync(0xffffffffu, a1, o);
                a2 += __shfl_xor_sync(0xffffffffu, a2, o);
            }
            if (lane == 0) {
                const float inv_k = 1.0f / (float)K;
                const float dm = a1 * inv_k;  // mean - c
                const float var = fmaxf(fmaf(-dm, dm, a2 * inv_k), 0.f);
                stats[row] = make_float2(c + dm, rsqrtf(var + eps));
            }
        }
    };
    while (row < M) {
        int nr = row, nhh = h + 1;
        if (nhh == nh) {
            nr = row + nwarps;
            nhh = 0;
        }
        if ((q & 1) == 0) {
            if (nr < M) load_half(B, x, nr, nhh, K, lane);
            sum_half(A);
        } else {
            if (nr < M) load_half(A, x, nr, nhh, K, lane);
            sum_half(B);
        }
        row = nr;
        h = nhh;
        ++q;
    }
}

cudaError_t launch_ln_stats(int dt, const void* x, int M, int K, float eps, void* stats, int pdl, int sms,
                            cudaStream_t stream) {
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
    float2* sp = static_cast<float2*>(stats);
    if (dt == DT_F16) return cudaLaunchKernelEx(&cfg, fl_ln_stats_kernel<DT_F16>, xp, M, K, eps, sp);
    return cudaLaunchKernelEx(&cfg, fl_ln_stats_kernel<DT_BF16>, xp, M, K, eps, sp);
}

}  // namespace fl
