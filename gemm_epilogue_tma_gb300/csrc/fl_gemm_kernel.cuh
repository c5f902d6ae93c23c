// Persistent, warp-specialised fused dense-layer kernel for sm_103a.
//
//   out[M, N] = epilogue( prologue(A)[M, K] * W[N, K]^T )
//
// One CTA per SM walks output tiles of 128 x BN. Roles inside a CTA:
//   warp 0        TMA producer: fills an S-stage ring of (A, W[, W2]) K-slices
//                 (64 elements = 128 B per row, 128-byte swizzle).
//   warp 1        TMEM owner and MMA issuer: one thread issues
//                 tcgen05.mma.cta_group::1.kind::f16 (128 x BN x 16) into an
//                 fp32 accumulator in tensor memory, double-buffered where the
//                 columns allow (the epilogue of a tile then overlaps the next
//                 tile's MMAs).
//   warps 4-7     (norm prologues only) transform warpgroup. With 128-wide
//                 tiles (one or two weights) thread t folds tile row t
//                 (RMS: x * gamma and sum(x^2); LayerNorm: (x - mean) * rstd
//                 * gamma + beta with the row statistics computed ahead of the
//                 GEMM) into a 32-column tensor-memory slot, and the MMA reads
//                 A from there; with 256-wide tiles the fold rewrites the
//                 staged operand in place.
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

#include "fl_common.cuh"
#include "fl_fold.cuh"

namespace fl {

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int DT, int BN, int PRO, bool DUAL, bool MULTI>
__global__ void __launch_bounds__(PRO != PRO_NONE ? 384 : 256, 1)
    fl_gemm_kernel(const __grid_constant__ ParamsT<MULTI> p) {
    using C = TileCfg<BN, DUAL>;
    using Ops = DTypeOps<DT>;
    constexpr int S = C::STAGES;
    constexpr int EPI_WARP0 = PRO != PRO_NONE ? 8 : 4;
    constexpr uint32_t IDESC = umma_idesc_f16(Ops::kFormat, kBM, BN);
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile width");
    // Norm prologue with one weight and a 128-wide tile: the folded activation
    // goes to tensor memory (one 32-column slot per stage after the two
    // accumulators) and the MMA reads it from there, which takes the fold's
    // shared-memory writes and the MMA's activation reads off shared memory.
    constexpr bool ATMEM = PRO != PRO_NONE && BN == 128;
    // accumulator buffers: two (the epilogue of a tile overlaps the next
    // tile's MMAs) unless the activation slots then no longer fit (the
    // gate/up kernel: 2 x 256 accumulator columns)
    constexpr int NBUF = 2 * C::ACC_COLS + (ATMEM ? 32 * S : 0) <= 512 ? 2 : 1;
    constexpr uint32_t TMEM_ALLOC = ATMEM ? 512u : (uint32_t)C::TMEM_COLS;
    constexpr uint32_t A_COL0 = (uint32_t)NBUF * C::ACC_COLS;
    static_assert(!ATMEM || A_COL0 + 32u * S <= 512u, "activation slots must fit in tensor memory");

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
        for (int i = 0; i < p.n_out; ++i) {
            tma_prefetch_desc(tm_b(p, i));
            tma_prefetch_desc(tm_out(p, i));
        }
        if (DUAL) tma_prefetch_desc(&p.tmB2);
        if (PRO != PRO_NONE) tma_prefetch_desc(&p.tmGamma);
        if (PRO == PRO_LN && p.beta != nullptr) tma_prefetch_desc(&p.tmBeta);
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, TMEM_ALLOC);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);
    // Everything above overlaps the previous kernel on the stream; every
    // global-memory access below waits for it. The L2 prefetch of the first
    // weight tiles may run early: L2 is the point of coherence, so it cannot
    // return stale data.
    if (warp == 0 && lane == 0 && blockIdx.x < p.num_tiles) {
        const OutSel o = out_sel(p, blockIdx.x / p.num_m_blocks);
        const int n0 = o.nb * BN;
        for (int kb = 0; kb < S && kb < nk; ++kb) {
            tma_prefetch_2d(tm_b(p, o.oi), kb * kBK, n0);
            if (DUAL) tma_prefetch_2d(&p.tmB2, kb * kBK, n0);
        }
    }
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();

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
                const OutSel o = out_sel(p, tile / p.num_m_blocks);
                const int n0 = o.nb * BN;
                const CUtensorMap* tb = tm_b(p, o.oi);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bar(empty_bar(s), ph ^ 1u, p.status, p.timeout_ns, 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), main_bytes);
                    tma_load_2d(stage_a(s), &p.tmA, full_bar(s), kb * kBK, m0);
                    tma_load_2d(stage_b(s), tb, full_bar(s), kb * kBK, n0);
                    if (DUAL) tma_load_2d(stage_b2(s), &p.tmB2, full_bar(s), kb * kBK, n0);
                    if (PRO != PRO_NONE) {
                        tma_load_2d(gb_slot(s), &p.tmGamma, full_bar(s), kb * kBK, 0);
                        if (PRO == PRO_LN && p.beta != nullptr)
                            tma_load_2d(gb_slot(s) + 128, &p.tmBeta, full_bar(s), kb * kBK, 0);
                    }
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
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
                const int buf = NBUF == 2 ? (it & 1) : 0;
                const uint32_t tph = NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
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
                        if (ATMEM) {
                            // 16 K elements = 8 columns of the stage's activation slot
                            const uint32_t ta = tmem_base + A_COL0 + 32u * s + 8u * kk;
                            umma_f16_ts(d, ta, db + 2 * kk, IDESC, (kb | kk) != 0);
                            if (DUAL) {
                                const uint64_t db2 = sw128_kmajor_desc(stage_b2(s));
                                umma_f16_ts(d + BN, ta, db2 + 2 * kk, IDESC, (kb | kk) != 0);
                            }
                            continue;
                        }
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
    } else if (ATMEM && warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ transform into TMEM
        const int t = threadIdx.x - 128;  // tile row = TMEM lane
        const uint32_t a_lane = (uint32_t)(32 * (warp & 3)) << 16;
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
            float rstd = 1.f, nmr = 0.f;  // LayerNorm: 1/std and -mean/std of row t
            float ss[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ss[i] = 0.f;
            if (PRO == PRO_LN) {
                const int row = (tile % p.num_m_blocks) * kBM + t;
                if (row < p.M) {
                    const float2 st = reinterpret_cast<const float2*>(p.ln_stats)[row];
                    rstd = st.y;
                    nmr = -st.x * st.y;
                }
            }
            for (int kb = 0; kb < nk; ++kb) {
                if (!wait_bar(full_bar(s), ph, p.status, p.timeout_ns, 6)) {
                    ok = false;
                    break;
                }
                uint32_t o[32];
                if (PRO == PRO_RMS) {
                    fold_rms_row<DT>(stage_a(s), gb_slot(s), t, ss, o);
                } else if (PRO == PRO_ADD) {
                    fold_add_row<DT>(stage_a(s), gb_slot(s), t, o);
                } else {
                    uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[0]);
                    uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[16]);
                    fold_ln_row<DT, 4, 0>(stage_a(s), gb_slot(s), p.beta != nullptr, t, rstd, nmr, lo);
                    fold_ln_row<DT, 4, 4>(stage_a(s), gb_slot(s), p.beta != nullptr, t, rstd, nmr, hi);
                }
                tmem_st_32x32b_x32(tmem_base + a_lane + A_COL0 + 32u * s, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xform_bar(s));
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (PRO == PRO_RMS) {
                const int buf = NBUF == 2 ? (it & 1) : 0;
                const uint32_t tph = NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
                if (!wait_bar(tempty_bar(buf), tph ^ 1u, p.status, p.timeout_ns, 7)) break;
                const float sum = ((ss[0] + ss[1]) + (ss[2] + ss[3])) + ((ss[4] + ss[5]) + (ss[6] + ss[7]));
                rowscale[buf * kBM + t] = rsqrtf(sum / (float)p.K + p.eps);
                __syncwarp();
                if (lane == 0) mbar_arrive(sready_bar(buf));
            }
        }
    } else if (PRO != PRO_NONE && warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ transform
        const int t = threadIdx.x - 128;
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
            float mean[8], rstd[8], ss[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                mean[i] = 0.f;
                rstd[i] = 1.f;
                ss[i] = 0.f;
            }
            if (PRO == PRO_LN) {
                // rows (t >> 3) + 16 i of the tile
                const int r0 = (tile % p.num_m_blocks) * kBM + (t >> 3);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (r0 + 16 * i < p.M) {
                        const float2 st = reinterpret_cast<const float2*>(p.ln_stats)[r0 + 16 * i];
                        mean[i] = st.x;
                        rstd[i] = st.y;
                    }
                }
            }
            for (int kb = 0; kb < nk; ++kb) {
                if (!wait_bar(full_bar(s), ph, p.status, p.timeout_ns, 6)) {
                    ok = false;
                    break;
                }
                // gamma (and beta) of this K block arrived with the stage; columns
                // past K are zero in x, gamma and beta, so they stay zero
                if (PRO == PRO_RMS)
                    fold_rms_stage<DT>(stage_a(s), gb_slot(s), t, 8, ss);
                else if (PRO == PRO_ADD)
                    fold_add_stage<DT>(stage_a(s), gb_slot(s), t, 8);
                else
                    fold_ln_stage<DT>(stage_a(s), gb_slot(s), p.beta != nullptr, t, 8, mean, rstd);
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
                const int buf = NBUF == 2 ? (it & 1) : 0;
                const uint32_t tph = NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
#pragma unroll
                for (int i = 0; i < 8; ++i) ss[i] = row_allreduce8(ss[i]);
                if (!wait_bar(tempty_bar(buf), tph ^ 1u, p.status, p.timeout_ns, 7)) break;
                if ((t & 7) == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        rowscale[buf * kBM + (t >> 3) + 16 * i] = rsqrtf(ss[i] / (float)p.K + p.eps);
                }
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
        const T* res = reinterpret_cast<const T*>(p.residual);
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int m0 = (tile % p.num_m_blocks) * kBM;
            const OutSel o = out_sel(p, tile / p.num_m_blocks);
            const int n0 = o.nb * BN;
            const int N = out_n(p, o.oi);
            const int act = out_act(p, o.oi);
            const T* bias = reinterpret_cast<const T*>(out_bias(p, o.oi));
            const int buf = NBUF == 2 ? (it & 1) : 0;
            const uint32_t tph = NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
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
            // 64-column chunks this warp stores (rows or columns past the
            // output are skipped); the accumulator goes back to the MMA right
            // after the last chunk's TMEM load
            int nchunks = 0;
            if (m0 + q * 32 < p.M)
                while (nchunks < BN / 64 && n0 + nchunks * 64 < N) ++nchunks;
            bool released = false;
            auto release_acc = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(buf));
                released = true;
            };
            {
                for (int c = 0; c < nchunks; ++c) {
                    const int col0 = n0 + c * 64;
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
                            if (h == 1 && c == nchunks - 1) release_acc();
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const float gt = __uint_as_float(acc[e]) * rs;
                                const float u = __uint_as_float(up[e]) * rs;
                                v[e] = act_apply(ACT_SILU, gt) * u;
                            }
                        } else {
                            tmem_ld_wait();
                            if (h == 1 && c == nchunks - 1) release_acc();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(acc[e]) * rs;
                            if (bias != nullptr) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (cbase + j * 8 < N) {
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
                            if (act != ACT_NONE) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) v[e] = act_apply(act, v[e]);
                            }
                            if (res != nullptr && row_ok) {
                                const T* rrow = res + (size_t)row * N;
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (cbase + j * 8 < N) {
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
                        if (h == 0) {
                            // the previous chunk's TMA store has read the staging buffer
                            if (lane == 0) bulk_wait_group_read<0>();
                            __syncwarp();
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
                        tma_store_2d(tm_out(p, o.oi), ebuf, col0, m0 + q * 32);
                        bulk_commit_group();
                    }
                }
            }
            if (!released) release_acc();
        }
        if (lane == 0) bulk_wait_group_read<0>();  // global writes complete with the grid
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_ALLOC);
    }
}

template <int DT, int BN, int PRO, bool DUAL, bool MULTI>
cudaError_t launch_gemm(const ParamsT<MULTI>& p, int grid, cudaStream_t stream) {
    using C = TileCfg<BN, DUAL>;
    auto kern = fl_gemm_kernel<DT, BN, PRO, DUAL, MULTI>;
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace fl
