// Persistent, warp-specialised fused dense-layer kernel for sm_103a.
//
//   out[M, N] = epilogue( prologue(A)[M, K] * W[N, K]^T )
//
// One CTA per SM walks output tiles of 128 x BN. Roles inside a CTA:
//   warp 0        TMA producer: fills an S-stage ring of (A, W[, W2]) K-slices
//                 (64 elements = 128 B per row, 128-byte swizzle).
//   warp 1        TMEM owner and MMA issuer: one thread issues
//                 tcgen05.mma.cta_group::1.kind::f16 (128 x BN x 16) into a
//                 double-buffered fp32 accumulator in tensor memory.
//   warps 4-7     (norm prologues only) transform warpgroup, thread t <-> tile
//                 row t: RMS accumulates sum(x^2) and folds gamma into the
//                 staged operand in place; LayerNorm first streams the row
//                 block once for mean / variance (Chan's pairwise merge), then
//                 writes (x - mean) * rstd * gamma + beta in place.
//   last 4 warps  epilogue: tcgen05.ld 32 columns at a time, row scale (RMS),
//                 bias, activation, residual, round, stage in 128B-swizzled
//                 shared memory, TMA store (which clips the ragged tails).
// With DUAL (SwiGLU gate/up) the staged activation tile feeds two weight
// tiles into two accumulators, and the epilogue writes silu(g) * u.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel records
// a status word, every role leaves its loop, in-flight copies and MMAs are
// drained with bounded waits, and TMEM is released before exit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fl_internal.h"
#include "fl_ptx.cuh"

namespace fl {

template <int DT>
struct DTypeOps;

template <>
struct DTypeOps<DT_F16> {
    static constexpr uint32_t kFormat = 0;
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        return __half22float2(*reinterpret_cast<__half2*>(&u));
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
};

template <>
struct DTypeOps<DT_BF16> {
    static constexpr uint32_t kFormat = 1;
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// Waits for the phase of parity `parity` of `bar`. Gives up (returns false)
// after timeout_ns, or early once another role has recorded a failure.
static __device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, int* status,
                                           unsigned long long timeout_ns, int where) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*reinterpret_cast<volatile int*>(status) != 0) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                atomicCAS(status, 0, kStatusTimeout | (where << 8));
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* status,
                                         unsigned long long timeout_ns, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, status, timeout_ns, where);
}

// Time-bounded only: used while draining after a failure.
static __device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, unsigned long long ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > ns) return false;
    }
    return true;
}

__device__ __forceinline__ float act_apply(int act, float v) {
    switch (act) {
        case ACT_GELU: {
            const float c = 0.7978845608028654f;  // sqrt(2 / pi)
            return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
        }
        case ACT_SILU:
            return v / (1.0f + __expf(-v));
        case ACT_RELU:
            return fmaxf(v, 0.0f);
        default:
            return v;
    }
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int DT, int BN, int PRO, bool DUAL>
__global__ void __launch_bounds__(PRO != PRO_NONE ? 384 : 256, 1)
    fl_gemm_kernel(const __grid_constant__ GemmParams p) {
    using C = TileCfg<BN, DUAL>;
    using Ops = DTypeOps<DT>;
    constexpr int S = C::STAGES;
    constexpr int EPI_WARP0 = PRO != PRO_NONE ? 8 : 4;
    constexpr uint32_t IDESC = umma_idesc_f16(Ops::kFormat, kBM, BN);
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile width");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw_addr);

    auto stage_a = [&](int s) { return sbase + s * C::STAGE_BYTES; };
    auto stage_b = [&](int s) { return sbase + s * C::STAGE_BYTES + C::A_BYTES; };
    auto stage_b2 = [&](int s) { return sbase + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES; };
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto xform_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (3 * S + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
    auto sready_bar = [&](int b) { return bar0 + 8u * (3 * S + 4 + b); };
    const uint32_t drain_bar = bar0 + 8u * (3 * S + 6);
    const uint32_t slot_addr = sbase + C::OFF_SLOT;
    float* rowscale = reinterpret_cast<float*>(smem + C::OFF_ROWSCALE);  // [2][128]
    auto gb_slot = [&](int s) { return sbase + C::OFF_GB + 256u * s; };  // gamma | beta slices

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nk = p.num_k_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(xform_bar(s), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);
            mbar_init(sready_bar(b), 4);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        if (DUAL) tma_prefetch_desc(&p.tmB2);
        tma_prefetch_desc(&p.tmOut);
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            const uint32_t main_bytes = C::STAGE_BYTES + (PRO != PRO_NONE ? 128u : 0u) +
                                        (PRO == PRO_LN && p.beta != nullptr ? 128u : 0u);
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const int m0 = (tile % p.num_m_blocks) * kBM;
                const int n0 = (tile / p.num_m_blocks) * BN;
                const int passes = PRO == PRO_LN ? 2 : 1;
                for (int pass = 0; ok && pass < passes; ++pass) {
                    const bool stats = PRO == PRO_LN && pass == 0;
                    for (int kb = 0; kb < nk; ++kb) {
                        if (!wait_bar(empty_bar(s), ph ^ 1u, p.status, p.timeout_ns, 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_bar(s), stats ? (uint32_t)C::A_BYTES : main_bytes);
                        tma_load_2d(stage_a(s), &p.tmA, full_bar(s), kb * kBK, m0);
                        if (!stats) {
                            tma_load_2d(stage_b(s), &p.tmB, full_bar(s), kb * kBK, n0);
                            if (DUAL) tma_load_2d(stage_b2(s), &p.tmB2, full_bar(s), kb * kBK, n0);
                            if (PRO != PRO_NONE) {
                                tma_load_2d(gb_slot(s), &p.tmGamma, full_bar(s), kb * kBK, 0);
                                if (PRO == PRO_LN && p.beta != nullptr)
                                    tma_load_2d(gb_slot(s) + 128, &p.tmBeta, full_bar(s), kb * kBK, 0);
                            }
                        }
                        ++issued;
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            // Drain: every load this thread issued lands before the CTA may exit.
            const int pending = issued < S ? issued : S;
            for (int i = 1; i <= pending; ++i) {
                int idx = issued - i;
                wait_bar_drain(full_bar(idx % S), (uint32_t)((idx / S) & 1), 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int buf = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (PRO == PRO_LN) {
                    // statistics pass: the transform warps read these stages; release them
                    for (int kb = 0; kb < nk; ++kb) {
                        if (!wait_bar(xform_bar(s), ph, p.status, p.timeout_ns, 2)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive(empty_bar(s));
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                }
                if (!wait_bar(tempty_bar(buf), tph ^ 1u, p.status, p.timeout_ns, 3)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * C::ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    const uint32_t rb = PRO != PRO_NONE ? xform_bar(s) : full_bar(s);
                    if (!wait_bar(rb, ph, p.status, p.timeout_ns, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = sw128_kmajor_desc(stage_a(s));
                    const uint64_t db = sw128_kmajor_desc(stage_b(s));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // +32 bytes per 16-element K step inside the swizzled row
                        umma_f16_ss(d, da + 2 * kk, db + 2 * kk, IDESC, (kb | kk) != 0);
                        if (DUAL) {
                            const uint64_t db2 = sw128_kmajor_desc(stage_b2(s));
                            umma_f16_ss(d + BN, da + 2 * kk, db2 + 2 * kk, IDESC, (kb | kk) != 0);
                        }
                    }
                    umma_commit(empty_bar(s));
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull_bar(buf));
            }
            // Drain: all MMAs issued by this thread complete before TMEM is released.
            umma_commit(drain_bar);
            wait_bar_drain(drain_bar, 0, 20000000ull);
        }
    } else if (PRO != PRO_NONE && warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ transform
        const int t = threadIdx.x - 128;  // tile row
        const int sw = t & 7;
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
            float mean = 0.f, rstd = 1.f, ss = 0.f;
            if (PRO == PRO_LN) {
                float n = 0.f, m2 = 0.f;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bar(full_bar(s), ph, p.status, p.timeout_ns, 5)) {
                        ok = false;
                        break;
                    }
                    const uint32_t row = stage_a(s) + t * 128;
                    const int valid = min(kBK, p.K - kb * kBK);  // multiple of 8
                    float xs[64];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 v = ld_shared_v4(row + ((j ^ sw) << 4));
                        float2 a = Ops::unpack(v.x), b = Ops::unpack(v.y), c = Ops::unpack(v.z),
                               e = Ops::unpack(v.w);
                        xs[j * 8 + 0] = a.x; xs[j * 8 + 1] = a.y; xs[j * 8 + 2] = b.x; xs[j * 8 + 3] = b.y;
                        xs[j * 8 + 4] = c.x; xs[j * 8 + 5] = c.y; xs[j * 8 + 6] = e.x; xs[j * 8 + 7] = e.y;
                    }
                    // out-of-range K columns are zero-filled by TMA: they add 0 to the sum,
                    // and are excluded from the deviation sum below by the count
                    float sum = 0.f;
#pragma unroll
                    for (int e = 0; e < 64; ++e) sum += xs[e];
                    const float cnt = (float)valid;
                    const float cm = sum / cnt;
                    float cm2 = 0.f;
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const float dlt = xs[e] - cm;
                        cm2 += (e < valid) ? dlt * dlt : 0.f;
                    }
                    const float nn = n + cnt;
                    const float delta = cm - mean;
                    mean += delta * (cnt / nn);
                    m2 += cm2 + delta * delta * (n * cnt / nn);
                    n = nn;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xform_bar(s));
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                rstd = rsqrtf(m2 / (float)p.K + p.eps);
            }
            for (int kb = 0; kb < nk; ++kb) {
                if (!wait_bar(full_bar(s), ph, p.status, p.timeout_ns, 6)) {
                    ok = false;
                    break;
                }
                // gamma (and beta) of this K block arrived with the stage; columns
                // past K are zero in x, gamma and beta, so they stay zero
                const uint32_t row = stage_a(s) + t * 128;
                const uint32_t gsl = gb_slot(s);
                uint4 xv[8], gv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) xv[j] = ld_shared_v4(row + ((j ^ sw) << 4));
#pragma unroll
                for (int j = 0; j < 8; ++j) gv[j] = ld_shared_v4(gsl + j * 16);
                if (PRO == PRO_RMS) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = Ops::unpack(xw[q]);
                            ss = fmaf(f.x, f.x, ss);
                            ss = fmaf(f.y, f.y, ss);
                        }
                        // the product of two 16-bit values rounded once: same as
                        // rounding the exact fp32 product
                        xv[j].x = Ops::mul2(xv[j].x, gv[j].x);
                        xv[j].y = Ops::mul2(xv[j].y, gv[j].y);
                        xv[j].z = Ops::mul2(xv[j].z, gv[j].z);
                        xv[j].w = Ops::mul2(xv[j].w, gv[j].w);
                    }
                } else {
                    uint4 bv[8];
                    const bool has_beta = p.beta != nullptr;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        bv[j] = has_beta ? ld_shared_v4(gsl + 128 + j * 16) : make_uint4(0u, 0u, 0u, 0u);
                    const float nb = -mean * rstd;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
                        const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
                        const uint32_t bw[4] = {bv[j].x, bv[j].y, bv[j].z, bv[j].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = Ops::unpack(xw[q]), g2 = Ops::unpack(gw[q]), b2 = Ops::unpack(bw[q]);
                            xw[q] = Ops::pack(fmaf(fmaf(f.x, rstd, nb), g2.x, b2.x),
                                              fmaf(fmaf(f.y, rstd, nb), g2.y, b2.y));
                        }
                        xv[j] = make_uint4(xw[0], xw[1], xw[2], xw[3]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) st_shared_v4(row + ((j ^ sw) << 4), xv[j].x, xv[j].y, xv[j].z, xv[j].w);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(xform_bar(s));
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (PRO == PRO_RMS) {
                // the row scale of buffer (it & 1) is free once the epilogue has
                // released that accumulator buffer for this tile
                const int buf = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (!wait_bar(tempty_bar(buf), tph ^ 1u, p.status, p.timeout_ns, 7)) break;
                rowscale[buf * kBM + t] = rsqrtf(ss / (float)p.K + p.eps);
                __syncwarp();
                if (lane == 0) mbar_arrive(sready_bar(buf));
            }
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter
        const uint32_t ebuf = sbase + C::OFF_EPI + q * C::EPI_BUF_BYTES;
        const uint32_t my_row_addr = ebuf + lane * 128;
        const int sw = lane & 7;
        int it = 0;
        using T = uint16_t;
        const T* bias = reinterpret_cast<const T*>(p.bias);
        const T* res = reinterpret_cast<const T*>(p.residual);
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int m0 = (tile % p.num_m_blocks) * kBM;
            const int n0 = (tile / p.num_m_blocks) * BN;
            const int buf = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            if (!wait_bar(tfull_bar(buf), tph, p.status, p.timeout_ns, 8)) break;
            tc_fence_after();
            float rs = 1.f;
            if (PRO == PRO_RMS) {
                if (!wait_bar(sready_bar(buf), tph, p.status, p.timeout_ns, 9)) break;
                rs = rowscale[buf * kBM + q * 32 + lane];
            }
            const int row = m0 + q * 32 + lane;
            const bool row_ok = row < p.M;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::ACC_COLS);
            if (m0 + q * 32 < p.M) {
                for (int c = 0; c < BN / 64; ++c) {
                    const int col0 = n0 + c * 64;
                    if (col0 >= p.N) break;
                    // staging buffer of this warp is reused: the previous store must have read it
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int cbase = col0 + h * 32;
                        uint32_t acc[32];
                        tmem_ld_32x32b_x32(tbase + c * 64 + h * 32, acc);
                        float v[32];
                        if (DUAL) {
                            uint32_t up[32];
                            tmem_ld_32x32b_x32(tbase + BN + c * 64 + h * 32, up);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const float gt = __uint_as_float(acc[e]) * rs;
                                const float u = __uint_as_float(up[e]) * rs;
                                v[e] = gt / (1.0f + __expf(-gt)) * u;
                            }
                        } else {
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(acc[e]) * rs;
                            if (bias != nullptr) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (cbase + j * 8 < p.N) {
                                        const uint4 bv = ldg_v4(bias + cbase + j * 8);
                                        const float2 b0 = Ops::unpack(bv.x), b1 = Ops::unpack(bv.y),
                                                     b2 = Ops::unpack(bv.z), b3 = Ops::unpack(bv.w);
                                        v[j * 8 + 0] += b0.x; v[j * 8 + 1] += b0.y;
                                        v[j * 8 + 2] += b1.x; v[j * 8 + 3] += b1.y;
                                        v[j * 8 + 4] += b2.x; v[j * 8 + 5] += b2.y;
                                        v[j * 8 + 6] += b3.x; v[j * 8 + 7] += b3.y;
                                    }
                                }
                            }
                            if (p.act != ACT_NONE) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) v[e] = act_apply(p.act, v[e]);
                            }
                            if (res != nullptr && row_ok) {
                                const T* rrow = res + (size_t)row * p.N;
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (cbase + j * 8 < p.N) {
                                        const uint4 rv = *reinterpret_cast<const uint4*>(rrow + cbase + j * 8);
                                        const float2 r0 = Ops::unpack(rv.x), r1 = Ops::unpack(rv.y),
                                                     r2 = Ops::unpack(rv.z), r3 = Ops::unpack(rv.w);
                                        v[j * 8 + 0] += r0.x; v[j * 8 + 1] += r0.y;
                                        v[j * 8 + 2] += r1.x; v[j * 8 + 3] += r1.y;
                                        v[j * 8 + 4] += r2.x; v[j * 8 + 5] += r2.y;
                                        v[j * 8 + 6] += r3.x; v[j * 8 + 7] += r3.y;
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int chunk = h * 4 + j;  // 16-byte chunk of the 128-byte row
                            st_shared_v4(my_row_addr + ((chunk ^ sw) << 4),
                                         Ops::pack(v[j * 8 + 0], v[j * 8 + 1]),
                                         Ops::pack(v[j * 8 + 2], v[j * 8 + 3]),
                                         Ops::pack(v[j * 8 + 4], v[j * 8 + 5]),
                                         Ops::pack(v[j * 8 + 6], v[j * 8 + 7]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmOut, ebuf, col0, m0 + q * 32);
                        bulk_commit_group();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
        if (lane == 0) bulk_wait_group<0>();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int DT, int BN, int PRO, bool DUAL>
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
    using C = TileCfg<BN, DUAL>;
    auto kern = fl_gemm_kernel<DT, BN, PRO, DUAL>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int threads = PRO != PRO_NONE ? 384 : 256;
    kern<<<grid, threads, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fl
