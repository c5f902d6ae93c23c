// Split-K fused dense-layer kernel for few output tiles (small-M decode
// shapes): a weight-streaming variant bound by HBM bandwidth.
//
// The grid holds tiles x splits CTAs; the `splits` CTAs of one 128 x BN output
// tile form a thread-block cluster and each takes one contiguous K range, so
// every weight byte is read from HBM exactly once across the grid. Inside a
// CTA the roles match the tile kernel (TMA producer, tcgen05 MMA issuer,
// norm transform warpgroup, TMEM reader); the activation box is only as tall
// as the real rows (M rounded up to 16), so a decode step stages little more
// than the weights.
//
// Reduction: each CTA drains its fp32 partial tile from TMEM into its own
// shared memory (with its partial RMS sum of squares), the cluster barrier
// publishes it, and every CTA then sums an interleaved slice of the tile over
// distributed shared memory (ld.shared::cluster), applies the epilogue (row
// scale, bias, activation, residual) and stores 16-byte vectors. No global
// scratch memory is used.
//
// LayerNorm needs the row statistics before the fold: the transform warps
// compute them at the start from the activation rows (two passes over L2,
// coalesced warp loads), which is cheap because the activation is small.
#pragma once

#include "fl_common.cuh"
#include "fl_fold.cuh"

namespace fl {

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int DT, int BN, int PRO>
__global__ void __launch_bounds__(PRO != PRO_NONE ? 384 : 256, 1)
    fl_splitk_kernel(const __grid_constant__ GemmParams p) {
    if (threadIdx.x == 0) FL_MARK(p, 0);
    using C = SplitCfg<BN>;
    using Ops = DTypeOps<DT>;
    constexpr int S = C::STAGES;
    constexpr int EPI_WARP0 = PRO != PRO_NONE ? 8 : 4;
    constexpr uint32_t IDESC = umma_idesc_f16(Ops::kFormat, kBM, BN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw_addr);

    auto stage_a = [&](int s) { return sbase + s * C::STAGE_BYTES; };
    auto stage_b = [&](int s) { return sbase + s * C::STAGE_BYTES + C::A_BYTES; };
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto xform_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    const uint32_t tfull_bar = bar0 + 8u * (3 * S);
    const uint32_t drain_bar = bar0 + 8u * (3 * S + 1);
    const uint32_t slot_addr = sbase + C::OFF_SLOT;
    float* ssbuf = reinterpret_cast<float*>(smem + C::OFF_SS);
    float2* lnstat = reinterpret_cast<float2*>(smem + C::OFF_LN);
    auto gb_slot = [&](int s) { return sbase + C::OFF_GB + 256u * s; };
    const uint32_t red_base = sbase;  // the ring, reused once the main loop is over

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int splits = p.splits;
    const int rank = (int)cluster_ctarank();
    const int tile = blockIdx.x / splits;
    const int m0 = (tile % p.num_m_blocks) * kBM;
    const int n0 = (tile / p.num_m_blocks) * BN;
    const int nk = p.num_k_blocks;
    const int kb0 = rank * p.kps;
    const int kb1 = min(nk, kb0 + p.kps);
    const int rows = min(kBM, p.M - m0);       // real rows of this tile
    const int box_rows = p.a_rows;             // rows the activation box stages
    const uint32_t a_bytes = (uint32_t)box_rows * 128u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(xform_bar(s), 4);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        if (PRO != PRO_NONE) tma_prefetch_desc(&p.tmGamma);
        if (PRO == PRO_LN && p.beta != nullptr) tma_prefetch_desc(&p.tmBeta);
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);
    // Everything above overlaps the previous kernel on the stream; every
    // global-memory access below waits for it, except the L2 prefetch of this
    // CTA's first weight tiles (L2 is the point of coherence).
    if (warp == 0 && lane == 0) {
        for (int kb = kb0; kb < kb0 + S && kb < kb1; ++kb) tma_prefetch_2d(&p.tmB, kb * kBK, n0);
    }
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
    if (threadIdx.x == 0) FL_MARK(p, 1);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            const uint32_t bytes = a_bytes + (uint32_t)C::B_BYTES + (PRO != PRO_NONE ? 128u : 0u) +
                                   (PRO == PRO_LN && p.beta != nullptr ? 128u : 0u);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bar(empty_bar(s), ph ^ 1u, p.status, p.timeout_ns, 21)) break;
                mbar_arrive_expect_tx(full_bar(s), bytes);
                tma_load_2d(stage_a(s), &p.tmA, full_bar(s), kb * kBK, m0);
                tma_load_2d(stage_b(s), &p.tmB, full_bar(s), kb * kBK, n0);
                if (PRO != PRO_NONE) {
                    tma_load_2d(gb_slot(s), &p.tmGamma, full_bar(s), kb * kBK, 0);
                    if (PRO == PRO_LN && p.beta != nullptr)
                        tma_load_2d(gb_slot(s) + 128, &p.tmBeta, full_bar(s), kb * kBK, 0);
                }
                if (issued == 0) FL_MARK(p, 2);
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            const int pending = issued < S ? issued : S;
            for (int i = 1; i <= pending; ++i) {
                const int idx = issued - i;
                wait_bar_drain(full_bar(idx % S), (uint32_t)((idx / S) & 1), 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                const uint32_t rb = PRO != PRO_NONE ? xform_bar(s) : full_bar(s);
                if (!wait_bar(rb, ph, p.status, p.timeout_ns, 22)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (kb == kb0) FL_MARK(p, 3);
                const uint64_t da = sw128_kmajor_desc(stage_a(s));
                const uint64_t db = sw128_kmajor_desc(stage_b(s));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_f16_ss(tmem_base, da + 2 * kk, db + 2 * kk, IDESC, (kb != kb0) || (kk != 0));
                umma_commit(empty_bar(s));
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) umma_commit(tfull_bar);
            FL_MARK(p, 4);
            umma_commit(drain_bar);
            wait_bar_drain(drain_bar, 0, 20000000ull);
        }
    } else if (PRO != PRO_NONE && warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ transform
        const int t = threadIdx.x - 128;
        const int ni = box_rows / 16;  // rows of this thread: t/8 + 16 i
        float mean[8], rstd[8], ss[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mean[i] = 0.f;
            rstd[i] = 1.f;
            ss[i] = 0.f;
        }
        if (PRO == PRO_LN) {
            // statistics of the whole row: warp w takes rows w, w + 4, ...
            const uint16_t* xg = reinterpret_cast<const uint16_t*>(p.a_ptr);
            for (int r = warp - 4; r < rows; r += 4) {
                const uint16_t* xr = xg + (size_t)(m0 + r) * p.K;
                float a = 0.f;
                for (int k = lane * 8; k < p.K; k += 256) {
                    const uint4 v = ldg_v4(xr + k);
                    const float2 f0 = Ops::unpack(v.x), f1 = Ops::unpack(v.y), f2 = Ops::unpack(v.z),
                                 f3 = Ops::unpack(v.w);
                    a += ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                }
                const float mu = warp_sum(a) / (float)p.K;
                float q = 0.f;
                for (int k = lane * 8; k < p.K; k += 256) {
                    const uint4 v = ldg_v4(xr + k);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = Ops::unpack(w4[e]);
                        q = fmaf(f.x - mu, f.x - mu, q);
                        q = fmaf(f.y - mu, f.y - mu, q);
                    }
                }
                const float var = warp_sum(q) / (float)p.K;
                if (lane == 0) lnstat[r] = make_float2(mu, rsqrtf(var + p.eps));
            }
            named_bar_sync(1, 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = (t >> 3) + 16 * i;
                if (i < ni && r < rows) {
                    const float2 st = lnstat[r];
                    mean[i] = st.x;
                    rstd[i] = st.y;
                }
            }
        }
        int s = 0;
        uint32_t ph = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_bar(full_bar(s), ph, p.status, p.timeout_ns, 23)) break;
            if (PRO == PRO_RMS)
                fold_rms_stage<DT>(stage_a(s), gb_slot(s), t, ni, ss);
            else
                fold_ln_stage<DT>(stage_a(s), gb_slot(s), p.beta != nullptr, t, ni, mean, rstd);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(xform_bar(s));
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (PRO == PRO_RMS) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float v = row_allreduce8(ss[i]);
                if ((t & 7) == 0 && i < ni) ssbuf[(t >> 3) + 16 * i] = v;
            }
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ TMEM -> shared partial
        const int q = warp & 3;
        const int r = q * 32 + lane;
        if (wait_bar(tfull_bar, 0, p.status, p.timeout_ns, 24)) {
            tc_fence_after();
            if (threadIdx.x == 32 * EPI_WARP0) FL_MARK(p, 5);
            if (q * 32 < rows) {
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
                const uint32_t dst = red_base + (uint32_t)(r * C::RED_STRIDE) * 4u;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, v);
                    tmem_ld_wait();
                    if (r < rows) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(dst + (c * 32 + j * 4) * 4, v[j * 4], v[j * 4 + 1], v[j * 4 + 2], v[j * 4 + 3]);
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) FL_MARK(p, 6);
    // partials of every CTA of the cluster are written and visible after this
    cluster_sync_all();
    if (threadIdx.x == 0) FL_MARK(p, 7);

    // ---------------------------------------------------------------- reduction + epilogue
    {
        const bool failed = *reinterpret_cast<volatile int*>(p.status) != 0;
        const int cpr = BN / 8;  // 8-column chunks per row
        const int items = rows * cpr;
        using T = uint16_t;
        const T* bias = reinterpret_cast<const T*>(p.bias);
        const T* res = reinterpret_cast<const T*>(p.residual);
        T* out = reinterpret_cast<T*>(p.out_ptr);
        for (int i = rank + splits * (int)threadIdx.x; !failed && i < items; i += splits * (int)blockDim.x) {
            const int row = i / cpr, chunk = i % cpr;
            const int col = n0 + chunk * 8;
            if (col >= p.N) continue;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            float ss = 0.f;
            const uint32_t off = red_base + (uint32_t)(row * C::RED_STRIDE + chunk * 8) * 4u;
            for (int qr = 0; qr < splits; ++qr) {
                const uint32_t a = mapa_shared(off, (uint32_t)qr);
                const float4 lo = ld_cluster_v4(a), hi = ld_cluster_v4(a + 16);
                v[0] += lo.x; v[1] += lo.y; v[2] += lo.z; v[3] += lo.w;
                v[4] += hi.x; v[5] += hi.y; v[6] += hi.z; v[7] += hi.w;
                if (PRO == PRO_RMS) ss += ld_cluster_f32(mapa_shared(smem_u32(ssbuf + row), (uint32_t)qr));
            }
            if (PRO == PRO_RMS) {
                const float rs = rsqrtf(ss / (float)p.K + p.eps);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] *= rs;
            }
            if (bias != nullptr) {
                const uint4 bv = ldg_v4(bias + col);
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 b2 = Ops::unpack(bw[e]);
                    v[2 * e] += b2.x;
                    v[2 * e + 1] += b2.y;
                }
            }
            if (p.act != ACT_NONE) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = act_apply(p.act, v[e]);
            }
            const size_t g = (size_t)(m0 + row) * p.N + col;
            if (res != nullptr) {
                const uint4 rv = *reinterpret_cast<const uint4*>(res + g);
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 r2 = Ops::unpack(rw[e]);
                    v[2 * e] += r2.x;
                    v[2 * e + 1] += r2.y;
                }
            }
            *reinterpret_cast<uint4*>(out + g) = make_uint4(Ops::pack(v[0], v[1]), Ops::pack(v[2], v[3]),
                                                             Ops::pack(v[4], v[5]), Ops::pack(v[6], v[7]));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) FL_MARK(p, 8);
    // no CTA leaves while a peer may still read its shared memory
    cluster_sync_all();
    if (threadIdx.x == 0) FL_MARK(p, 9);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// How many clusters of `splits` CTAs of this kernel can be resident at once.
template <int DT, int BN, int PRO>
int splitk_max_clusters(int splits) {
    using C = SplitCfg<BN>;
    auto kern = fl_splitk_kernel<DT, BN, PRO>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, 1, 1);
    cfg.blockDim = dim3(PRO != PRO_NONE ? 384 : 256, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int DT, int BN, int PRO>
cudaError_t launch_splitk(const GemmParams& p, int grid, int splits, cudaStream_t stream) {
    using C = SplitCfg<BN>;
    auto kern = fl_splitk_kernel<DT, BN, PRO>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(PRO != PRO_NONE ? 384 : 256, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = p.pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace fl
