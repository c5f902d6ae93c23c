// Decode kernels for one to four activation rows: the dense layer as a
// weight-streaming matrix-vector product on the CUDA cores, and the whole
// SwiGLU FFN block in one launch.
//
// With M <= 4 rows a 128-row tensor-core MMA is more than 97 % padding and the
// step is bound by reading the weights once from HBM; what decides its time
// is how early the weight stream starts and how little fixed work surrounds
// it. Here every CTA builds the prologue-transformed activation rows in
// shared memory (RMSNorm / LayerNorm statistics of the few rows, then the
// fold, rounded once to the dtype as in the tensor-core kernels), and every
// warp streams whole weight rows with 16-byte loads, keeps one fp32 partial
// dot product per activation row, adds them across the warp with a fixed
// butterfly and applies the epilogue (row scale, bias, activation, residual).
// No reduction crosses a warp, so there is no cluster, no tensor memory and
// no exchange. Weight rows are dealt to warps round-robin over the grid, CTA
// by CTA, so every SM streams the same number of bytes to within one row, and
// each warp keeps two rows' loads in flight.
//
// The FFN kernel runs the gate/up product (h = silu(g) * u, rounded once),
// then a grid-wide barrier, then the down projection with the residual, in
// one launch: h goes to the caller's workspace and is read back through L2,
// never waiting on a second launch. Its grid is sized so every CTA is
// resident, and it lets the next kernel on the stream in only after the
// barrier, so a dependent grid cannot take the slots its CTAs need. Every
// wait is bounded.
#include "fl_common.cuh"
#include "fl_internal.h"

namespace fl {

namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kVec = 8;                 // 16-bit elements per 16-byte vector

// Rows of the prologue-transformed activation, in shared memory: xs[m][k],
// M <= MAXM rows of K 16-bit values; rscale[m] = the RMS row scale (else 1).
// Every thread loads its share of the raw rows at once (one memory round
// trip), the row statistics are added in a fixed order (per-thread partials,
// warp butterflies, then the warps in index order), and the fold rewrites the
// rows in place in shared memory.
template <int DT, int PRO, int MAXM>
__device__ void build_rows(const GemvParams& p, uint16_t* xs, float* rscale) {
    using Ops = DTypeOps<DT>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = p.M, K = p.K, kv = K / kVec, vecs = M * kv;
    __shared__ float part[kGemvWarps][MAXM][2];
    __shared__ float st_mean[MAXM], st_rstd[MAXM];
    // LayerNorm shifts each row by the mean of its first eight values
    float c[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        c[m] = 0.f;
        if (PRO == PRO_LN && m < M) {
            const uint4 h = ldg_v4(p.x + (size_t)m * K);
            const float2 a = Ops::unpack(h.x), b = Ops::unpack(h.y), d = Ops::unpack(h.z), e = Ops::unpack(h.w);
            c[m] = (((a.x + a.y) + (b.x + b.y)) + ((d.x + d.y) + (e.x + e.y))) * 0.125f;
        }
    }
    float s1[MAXM], s2[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) s1[m] = s2[m] = 0.f;
    constexpr int U = 4;
    for (int i0 = threadIdx.x; i0 < vecs; i0 += U * kGemvThreads) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * kGemvThreads;
            if (i < vecs) v[u] = ldg_v4(p.x + (size_t)(i / kv) * K + (size_t)(i % kv) * kVec);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * kGemvThreads;
            if (i < vecs) {
                const int m = i / kv;
                *reinterpret_cast<uint4*>(xs + (size_t)m * K + (size_t)(i % kv) * kVec) = v[u];
                if (PRO == PRO_RMS || PRO == PRO_LN) {
                    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int mm = 0; mm < MAXM; ++mm) {
                        if (mm == m) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = Ops::unpack(w[e]);
                                const float d0 = f.x - c[mm], d1 = f.y - c[mm];
                                s1[mm] += d0 + d1;
                                s2[mm] = fmaf(d0, d0, fmaf(d1, d1, s2[mm]));
                            }
                        }
                    }
                }
            }
        }
    }
    if (PRO == PRO_RMS || PRO == PRO_LN) {
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s1[m] += __shfl_xor_sync(0xffffffffu, s1[m], o);
                s2[m] += __shfl_xor_sync(0xffffffffu, s2[m], o);
            }
            if (lane == 0) {
                part[warp][m][0] = s1[m];
                part[warp][m][1] = s2[m];
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < MAXM) {
        const int m = threadIdx.x;
        float a1 = 0.f, a2 = 0.f;
        if (PRO == PRO_RMS || PRO == PRO_LN)
            for (int w = 0; w < kGemvWarps; ++w) {
                a1 += part[w][m][0];
                a2 += part[w][m][1];
            }
        const float inv_k = 1.0f / (float)K;
        rscale[m] = PRO == PRO_RMS ? rsqrtf(a2 * inv_k + p.eps) : 1.f;
        if (PRO == PRO_LN) {
            const float d = a1 * inv_k;
            st_mean[m] = c[m] + d;
            st_rstd[m] = rsqrtf(fmaxf(fmaf(-d, d, a2 * inv_k), 0.f) + p.eps);
        }
    }
    __syncthreads();
    // the fold, in place, rounded once to the dtype
    if (PRO != PRO_NONE) {
        for (int i = threadIdx.x; i < vecs; i += kGemvThreads) {
            const int m = i / kv, k = (i % kv) * kVec;
            uint4* slot = reinterpret_cast<uint4*>(xs + (size_t)m * K + k);
            const uint4 v = *slot;
            const uint4 g = ldg_v4(p.gamma + k);
            uint4 o;
            if (PRO == PRO_RMS) {
                o = make_uint4(Ops::mul2(v.x, g.x), Ops::mul2(v.y, g.y), Ops::mul2(v.z, g.z), Ops::mul2(v.w, g.w));
            } else if (PRO == PRO_ADD) {
                o = make_uint4(Ops::add2(v.x, g.x), Ops::add2(v.y, g.y), Ops::add2(v.z, g.z), Ops::add2(v.w, g.w));
            } else {
                const uint4 b = p.beta != nullptr ? ldg_v4(p.beta + k) : make_uint4(0u, 0u, 0u, 0u);
                const float mean = st_mean[m], rstd = st_rstd[m];
                const uint32_t xw[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w},
                               bw[4] = {b.x, b.y, b.z, b.w};
                uint32_t ow[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Ops::unpack(xw[e]), gg = Ops::unpack(gw[e]), bb = Ops::unpack(bw[e]);
                    ow[e] = Ops::pack(fmaf((f.x - mean) * rstd, gg.x, bb.x), fmaf((f.y - mean) * rstd, gg.y, bb.y));
                }
                o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
            *slot = o;
        }
        __syncthreads();
    }
}

// Two weight rows at once (a and b; b may be null): acc_a[m] += xs[m] . a and
// acc_b[m] += xs[m] . b over this lane's part of the K values, lanes taking
// 16-byte vectors at a 512-byte stride, both rows' loads of a chunk issued
// before any is used (2 x kChunk2 vectors in flight per lane).
constexpr int kChunk2 = 8;

template <int DT, int MAXM>
__device__ __forceinline__ void fma_vec(const uint4& wv, const uint16_t* xs, int M, int K, int k, float (&acc)[MAXM]) {
    using Ops = DTypeOps<DT>;
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    float2 wf[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) wf[e] = Ops::unpack(ww[e]);
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
        if (m < M) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)m * K + k);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xf = Ops::unpack(xw[e]);
                acc[m] = fmaf(xf.x, wf[e].x, fmaf(xf.y, wf[e].y, acc[m]));
            }
        }
    }
}

template <int DT, int MAXM>
__device__ __forceinline__ void dot_rows2(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                                          const uint16_t* xs, int M, int K, int lane, float (&acc_a)[MAXM],
                                          float (&acc_b)[MAXM]) {
    for (int k0 = lane * kVec; k0 < K; k0 += 32 * kVec * kChunk2) {
        uint4 va[kChunk2], vb[kChunk2];
#pragma unroll
        for (int u = 0; u < kChunk2; ++u) {
            const int k = k0 + u * 32 * kVec;
            if (k < K) {
                va[u] = ldg_v4(a + k);
                if (b != nullptr) vb[u] = ldg_v4(b + k);
            }
        }
#pragma unroll
        for (int u = 0; u < kChunk2; ++u) {
            const int k = k0 + u * 32 * kVec;
            if (k < K) {
                fma_vec<DT, MAXM>(va[u], xs, M, K, k, acc_a);
                if (b != nullptr) fma_vec<DT, MAXM>(vb[u], xs, M, K, k, acc_b);
            }
        }
    }
}

template <int MAXM>
__device__ __forceinline__ void warp_allreduce(float (&acc)[MAXM]) {
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
}

// L2 prefetch of the start of a weight row (before the dependency wait:
// weights are not written by the previous kernel, and L2 is the point of
// coherence, so the prefetch cannot bring in stale data).
__device__ __forceinline__ void prefetch_row(const uint16_t* w, int K, int lane) {
    const int bytes = K * 2;
    for (int off = lane * 128; off < bytes && off < 32 * 128 * 2; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(w) + off));
}

template <int DT, int PRO, int MAXM>
__global__ void __launch_bounds__(kGemvThreads) fl_gemv_kernel(const __grid_constant__ GemvParams p) {
    using Ops = DTypeOps<DT>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    __shared__ float rscale[MAXM];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // warp-major numbering: consecutive rows go to different CTAs, so every SM
    // gets the same number of rows to within one
    const int gw = warp * gridDim.x + blockIdx.x, nw = gridDim.x * kGemvWarps;
    const int rows = p.row0[p.n_out];
    auto row_of = [&](int r, int& oi, int& n) {
        oi = 0;
#pragma unroll
        for (int i = 1; i < 4; ++i)
            if (i < p.n_out && r >= p.row0[i]) oi = i;
        n = r - p.row0[oi];
    };
    if (gw < rows) {
        int oi, n;
        row_of(gw, oi, n);
        prefetch_row(p.W[oi] + (size_t)n * p.K, p.K, lane);
    }
    griddep_wait();
    build_rows<DT, PRO, MAXM>(p, xs, rscale);
    griddep_launch_dependents();
    // lane m finishes output row m of weight row r
    auto finish = [&](int r, const float (&acc)[MAXM]) {
        int oi, n;
        row_of(r, oi, n);
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (lane == m && m < p.M) {
                float v = acc[m] * rscale[m];
                if (p.bias[oi] != nullptr) v += Ops::unpack(p.bias[oi][n] | 0u).x;
                v = act_apply(p.act[oi], v);
                if (p.residual != nullptr) v += Ops::unpack(p.residual[(size_t)m * p.N[oi] + n] | 0u).x;
                const uint32_t packed = Ops::pack(v, 0.f);
                p.out[oi][(size_t)m * p.N[oi] + n] = (uint16_t)(packed & 0xffffu);
            }
        }
    };
    // two of this warp's rows per pass (r and r + nw), loads of both in flight
    for (int r = gw; r < rows; r += 2 * nw) {
        const int r2 = r + nw;
        int oi, n, oi2 = 0, n2 = 0;
        row_of(r, oi, n);
        if (r2 < rows) row_of(r2, oi2, n2);
        float acc[MAXM], acc2[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) acc[m] = acc2[m] = 0.f;
        dot_rows2<DT, MAXM>(p.W[oi] + (size_t)n * p.K, r2 < rows ? p.W[oi2] + (size_t)n2 * p.K : nullptr, xs, p.M,
                            p.K, lane, acc, acc2);
        warp_allreduce<MAXM>(acc);
        finish(r, acc);
        if (r2 < rows) {
            warp_allreduce<MAXM>(acc2);
            finish(r2, acc2);
        }
    }
}

// ---------------------------------------------------------------------------
// the SwiGLU FFN block in one launch
// ---------------------------------------------------------------------------
// Bounded grid barrier on a counter the host zeroed before the launch.
__device__ bool grid_barrier(unsigned int* counter, unsigned int expected, int* status,
                             unsigned long long timeout_ns) {
    __syncthreads();
    bool ok = true;
    __shared__ int bar_ok;
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's h is visible before it is counted
        atomicAdd(counter, 1u);
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            if (*reinterpret_cast<volatile unsigned int*>(counter) >= expected) break;
            if ((i & 63) == 0) {
                if (*reinterpret_cast<volatile int*>(status) != 0 || globaltimer_ns() - t0 > timeout_ns) {
                    atomicCAS(status, 0, kStatusTimeout | (60 << 8));
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();  // every CTA's h is visible to the reads below
        bar_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return bar_ok != 0;
}

template <int DT, int MAXM>
__global__ void __launch_bounds__(kGemvThreads) fl_ffn_decode_kernel(const __grid_constant__ FfnDecodeParams q) {
    using Ops = DTypeOps<DT>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    __shared__ float rscale[MAXM];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // warp-major numbering: consecutive rows go to different CTAs, so every SM
    // gets the same number of rows to within one
    const int gw = warp * gridDim.x + blockIdx.x, nw = gridDim.x * kGemvWarps;
    const int M = q.M, D = q.D, F = q.F;
    if (gw < F) {
        prefetch_row(q.Wg + (size_t)gw * D, D, lane);
        prefetch_row(q.Wu + (size_t)gw * D, D, lane);
    }
    griddep_wait();
    // phase 1: h = silu(xs Wg^T * rs) * (xs Wu^T * rs), xs = x * gamma
    {
        GemvParams p = {};
        p.x = q.x;
        p.gamma = q.gamma;
        p.M = M;
        p.K = D;
        p.eps = q.eps;
        build_rows<DT, PRO_RMS, MAXM>(p, xs, rscale);
    }
    for (int f = gw; f < F; f += nw) {
        float g[MAXM], u[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) g[m] = u[m] = 0.f;
        dot_rows2<DT, MAXM>(q.Wg + (size_t)f * D, q.Wu + (size_t)f * D, xs, M, D, lane, g, u);
        warp_allreduce<MAXM>(g);
        warp_allreduce<MAXM>(u);
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (lane == m && m < M) {
                const float v = act_apply(ACT_SILU, g[m] * rscale[m]) * (u[m] * rscale[m]);
                q.h[(size_t)m * F + f] = (uint16_t)(Ops::pack(v, 0.f) & 0xffffu);
            }
        }
    }
    const bool ok = grid_barrier(q.counter, gridDim.x, q.status, q.timeout_ns);
    // every CTA is resident and past phase 1: the next kernel may be scheduled
    griddep_launch_dependents();
    if (!ok) return;
    // phase 2: out = h Wd^T (+ bias_down) + x, h staged from L2 (not L1: it was
    // written by other SMs during this launch)
    {
        // h is M * F / 8 vectors: every thread's share issued at once
        const int hv = M * (F / kVec);
        constexpr int U = 8;
        for (int i0 = threadIdx.x; i0 < hv; i0 += U * kGemvThreads) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (i0 + u * kGemvThreads < hv)
                    v[u] = __ldcg(reinterpret_cast<const uint4*>(q.h) + i0 + u * kGemvThreads);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (i0 + u * kGemvThreads < hv) reinterpret_cast<uint4*>(xs)[i0 + u * kGemvThreads] = v[u];
        }
    }
    __syncthreads();
    auto finish = [&](int d, const float (&acc)[MAXM]) {
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (lane == m && m < M) {
                float v = acc[m];
                if (q.bias_down != nullptr) v += Ops::unpack(q.bias_down[d] | 0u).x;
                v += Ops::unpack(q.x[(size_t)m * D + d] | 0u).x;
                q.out[(size_t)m * D + d] = (uint16_t)(Ops::pack(v, 0.f) & 0xffffu);
            }
        }
    };
    for (int d = gw; d < D; d += 2 * nw) {
        const int d2 = d + nw;
        float acc[MAXM], acc2[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) acc[m] = acc2[m] = 0.f;
        dot_rows2<DT, MAXM>(q.Wd + (size_t)d * F, d2 < D ? q.Wd + (size_t)d2 * F : nullptr, xs, M, F, lane, acc, acc2);
        warp_allreduce<MAXM>(acc);
        finish(d, acc);
        if (d2 < D) {
            warp_allreduce<MAXM>(acc2);
            finish(d2, acc2);
        }
    }
}

template <int DT, int PRO, int MAXM>
cudaError_t gemv_launch(const GemvParams& p, int grid, int smem, int pdl, cudaStream_t stream) {
    auto kern = fl_gemv_kernel<DT, PRO, MAXM>;
    static cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemMax);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[0].val.programmaticStreamSerializationAllowed = pdl;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT, int MAXM>
cudaError_t ffn_launch(const FfnDecodeParams& q, int grid, int smem, int pdl, cudaStream_t stream) {
    auto kern = fl_ffn_decode_kernel<DT, MAXM>;
    static cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemMax);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[0].val.programmaticStreamSerializationAllowed = pdl;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, q);
}

template <typename Kern>
int resident_ctas(Kern kern, int smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemMax) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kGemvThreads, (size_t)smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

cudaError_t launch_gemv(int dt, int pro, const GemvParams& p, int sms, int pdl, cudaStream_t stream) {
    const int smem = p.M * p.K * 2;
    if (p.M < 1 || p.M > kGemvMaxRows || smem > kGemvSmemMax) return cudaErrorInvalidValue;
    // enough warps to deal the weight rows out evenly, at most two waves' worth of CTAs per SM
    const int rows = p.row0[p.n_out];
    int per_sm = 0;
#define FL_OCC(DT, PRO) \
    if (dt == DT && pro == PRO) per_sm = resident_ctas(fl_gemv_kernel<DT, PRO, kGemvMaxRows>, smem);
    FL_OCC(0, 0) FL_OCC(0, 1) FL_OCC(0, 2) FL_OCC(0, 3) FL_OCC(1, 0) FL_OCC(1, 1) FL_OCC(1, 2) FL_OCC(1, 3)
#undef FL_OCC
    if (per_sm < 1) return cudaErrorInvalidValue;
    if (per_sm > 4) per_sm = 4;
    int grid = sms * per_sm;
    const int need = (rows + kGemvWarps - 1) / kGemvWarps;
    if (grid > need) grid = need;
    const bool small = p.M <= 2;
#define FL_CASE(DT, PRO)                                                                              \
    if (dt == DT && pro == PRO)                                                                     \
        return small ? gemv_launch<DT, PRO, 2>(p, grid, smem, pdl, stream)                           \
                     : gemv_launch<DT, PRO, kGemvMaxRows>(p, grid, smem, pdl, stream);
    FL_CASE(0, 0) FL_CASE(0, 1) FL_CASE(0, 2) FL_CASE(0, 3) FL_CASE(1, 0) FL_CASE(1, 1) FL_CASE(1, 2) FL_CASE(1, 3)
#undef FL_CASE
    return cudaErrorInvalidValue;
}

int ffn_decode_grid(int dt, int M, int D, int F, int sms) {
    const int smem = M * (D > F ? D : F) * 2;
    if (M < 1 || M > kGemvMaxRows || smem > kGemvSmemMax) return 0;
    int per_sm = dt == 0 ? resident_ctas(fl_ffn_decode_kernel<0, kGemvMaxRows>, smem)
                         : resident_ctas(fl_ffn_decode_kernel<1, kGemvMaxRows>, smem);
    if (per_sm < 1) return 0;
    if (per_sm > 4) per_sm = 4;
    return sms * per_sm;  // every CTA resident at once: the grid barrier needs it
}

cudaError_t launch_ffn_decode(int dt, const FfnDecodeParams& q, int grid, int pdl, cudaStream_t stream) {
    const int smem = q.M * (q.D > q.F ? q.D : q.F) * 2;
    const bool small = q.M <= 2;
    if (dt == 0)
        return small ? ffn_launch<0, 2>(q, grid, smem, pdl, stream) : ffn_launch<0, kGemvMaxRows>(q, grid, smem, pdl, stream);
    return small ? ffn_launch<1, 2>(q, grid, smem, pdl, stream) : ffn_launch<1, kGemvMaxRows>(q, grid, smem, pdl, stream);
}

}  // namespace fl
