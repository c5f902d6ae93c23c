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
// Reduction: rank r of the cluster owns a slice of the tile's columns. Once
// its MMAs are done, a CTA tells its peers that its ring is free, drains its
// fp32 partial tile from TMEM into per-owner slots (with its partial RMS sum
// of squares per row), and sends each peer's slot with one bulk copy into
// that peer's ring (completion counted in bytes on the peer's barrier). Each
// owner then sums the `splits` partials of its slice from its own shared
// memory, applies the epilogue (row scale, bias, activation, residual) and
// stores 16-byte vectors. No global scratch memory is used, and the only
// cluster-wide barrier is split: arrived at once a CTA's incoming data is
// in, waited on just before exit, so no CTA leaves while a peer may still
// read or write its shared memory.
//
// LayerNorm folds with row statistics computed once per call by a separate
// small kernel (read here after the programmatic dependency resolves).
//
// DUAL (SwiGLU gate/up at decode sizes): each stage carries a tile of Wg and
// one of Wu, two accumulators are exchanged together, and the owner writes
// h = silu(gate / rms) * (up / rms).
#pragma once

#include "fl_common.cuh"
#include "fl_fold.cuh"

namespace fl {

// Warp roles: 0 TMA producer, 1 MMA issuer, then four transform warps (norm
// prologues; idle pair otherwise), then four epilogue warps (warp w reads
// TMEM lanes 32 (w % 4) ...). Every warp joins the final reduction. Ten warps
// at under 100 registers leave room for two CTAs per SM.
template <int PRO>
constexpr int splitk_threads() { return PRO != PRO_NONE ? 320 : 256; }

template <int DT, int BN, int PRO, bool DUAL, bool MULTI>
__global__ void __launch_bounds__(splitk_threads<PRO>(), 2)
    fl_splitk_kernel(const __grid_constant__ ParamsT<MULTI> p) {
    if (threadIdx.x == 0) FL_MARK(p, 0);
    using C = SplitCfg<BN, DUAL>;
    static_assert(!DUAL || PRO == PRO_RMS, "the gate/up kernel has the RMS prologue");
    using Ops = DTypeOps<DT>;
    constexpr int S = C::MAX_STAGES;  // barrier slots; the ring uses p.s_stages of them
    constexpr int XF_WARP0 = 2;
    constexpr int EPI_WARP0 = PRO != PRO_NONE ? 6 : 4;
    constexpr uint32_t IDESC = umma_idesc_f16(Ops::kFormat, kBM, BN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw_addr);

    const int box_rows = p.a_rows;             // rows the activation box stages
    const uint32_t a_bytes = (uint32_t)box_rows * 128u;
    const int NS = p.s_stages;
    const uint32_t ring = sbase + C::OFF_RING;
    const uint32_t stage_bytes = (uint32_t)p.s_stage_bytes;
    auto stage_a = [&](int s) { return ring + (uint32_t)s * stage_bytes; };
    auto stage_b = [&](int s) { return ring + (uint32_t)s * stage_bytes + a_bytes; };
    auto stage_b2 = [&](int s) { return ring + (uint32_t)s * stage_bytes + a_bytes + (uint32_t)C::B_BYTES; };
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto xform_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    const uint32_t tfull_bar = bar0 + 8u * (3 * S);
    const uint32_t drain_bar = bar0 + 8u * (3 * S + 1);
    const uint32_t peerfree_bar = bar0 + 8u * (3 * S + 2);  // every peer's ring may take my partials
    const uint32_t recvd_bar = bar0 + 8u * (3 * S + 3);     // every peer's partial of my slice is here
    const uint32_t slot_addr = sbase + C::OFF_SLOT;
    float* ssbuf = reinterpret_cast<float*>(smem + C::OFF_SS);
    auto gb_slot = [&](int s) { return sbase + C::OFF_GB + 256u * s; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int splits = p.splits;
    const int rank = (int)cluster_rank();
    const int tile = blockIdx.x / splits;
    const int m0 = (tile % p.num_m_blocks) * kBM;
    const OutSel osel = out_sel(p, tile / p.num_m_blocks);
    const int n0 = osel.nb * BN;
    const CUtensorMap* tmB = tm_b(p, osel.oi);
    const int nk = p.num_k_blocks;
    const int kb0 = rank * p.kps;
    const int kb1 = min(nk, kb0 + p.kps);
    const int rows = min(kBM, p.M - m0);       // real rows of this tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(xform_bar(s), 4);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        mbar_init(peerfree_bar, splits > 1 ? splits - 1 : 1);
        mbar_init(recvd_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(tmB);
        if (DUAL) tma_prefetch_desc(&p.tmB2);
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
    // first half of the barrier that makes every CTA's barriers exist before
    // a peer signals them (published by fence.mbarrier_init); its wait comes
    // right before the first remote access
    cluster_arrive_relaxed();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);
    // Everything above overlaps the previous kernel on the stream; global
    // memory is read only after it, with two exceptions for the weights:
    // with preload allowed (the caller guarantees that kernel does not write
    // W), the first ring stages' weight tiles go straight into shared memory
    // (the stage barrier expects the whole stage, so the MMA still waits for
    // the activation tile loaded after the dependency); else, when this CTA
    // has the SM to itself, an L2 prefetch of those tiles (L2 is the point of
    // coherence). With two CTAs per SM the prefetch would compete with the
    // previous kernel's stream for lines it then loses.
    const int npre = p.w_preload ? min(NS, kb1 - kb0) : 0;
    const uint32_t stage_tx = a_bytes + (uint32_t)C::STAGE_B_BYTES + (PRO != PRO_NONE ? 128u : 0u) +
                              (PRO == PRO_LN && p.beta != nullptr ? 128u : 0u);
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(full_bar(i), stage_tx);
            tma_load_2d(stage_b(i), tmB, full_bar(i), (kb0 + i) * kBK, n0);
            if (DUAL) tma_load_2d(stage_b2(i), &p.tmB2, full_bar(i), (kb0 + i) * kBK, n0);
        }
        if (p.s_one_per_sm)
            for (int kb = kb0 + npre; kb < kb0 + NS && kb < kb1; ++kb) {
                tma_prefetch_2d(tmB, kb * kBK, n0);
                if (DUAL) tma_prefetch_2d(&p.tmB2, kb * kBK, n0);
            }
    }
    griddep_wait();
    // The next kernel may launch now when its CTAs can only use idle SMs; with
    // two CTAs per SM it launches once this CTA's weight stream is over (see
    // the MMA issuer), so its early weight loads fill the tail of this one
    // instead of competing with its main loop.
    if (threadIdx.x == 0 && p.s_one_per_sm) griddep_launch_dependents();
    if (threadIdx.x == 0) FL_MARK(p, 1);

    bool ring_idle = false;  // MMA thread: every MMA of this CTA has completed
    __shared__ int xchg_ok;  // every partial of my slice is in (epilogue lead)
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (kb - kb0 >= npre) {  // a preloaded stage is fresh and already expects its bytes
                    if (!wait_bar(empty_bar(s), ph ^ 1u, p.status, p.timeout_ns, 21)) break;
                    mbar_arrive_expect_tx(full_bar(s), stage_tx);
                    tma_load_2d(stage_b(s), tmB, full_bar(s), kb * kBK, n0);
                    if (DUAL) tma_load_2d(stage_b2(s), &p.tmB2, full_bar(s), kb * kBK, n0);
                }
                tma_load_2d(stage_a(s), &p.tmA, full_bar(s), kb * kBK, m0);
                if (PRO != PRO_NONE) {
                    tma_load_2d(gb_slot(s), &p.tmGamma, full_bar(s), kb * kBK, 0);
                    if (PRO == PRO_LN && p.beta != nullptr)
                        tma_load_2d(gb_slot(s) + 128, &p.tmBeta, full_bar(s), kb * kBK, 0);
                }
                if (issued == 0) FL_MARK(p, 2);
                ++issued;
                if (++s == NS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            const int pending = issued < NS ? issued : NS;
            for (int i = 1; i <= pending; ++i) {
                const int idx = issued - i;
                wait_bar_drain(full_bar(idx % NS), (uint32_t)((idx / NS) & 1), 20000000ull);
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
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    umma_f16_ss(tmem_base, da + 2 * kk, db + 2 * kk, IDESC, (kb != kb0) || (kk != 0));
                    if (DUAL)
                        umma_f16_ss(tmem_base + BN, da + 2 * kk, sw128_kmajor_desc(stage_b2(s)) + 2 * kk, IDESC,
                                    (kb != kb0) || (kk != 0));
                }
                umma_commit(empty_bar(s));
                if (++s == NS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) umma_commit(tfull_bar);
            FL_MARK(p, 4);
            umma_commit(drain_bar);
            ring_idle = wait_bar_drain(drain_bar, 0, 20000000ull) && ok;
            if (!p.s_one_per_sm) griddep_launch_dependents();
        }
    } else if (PRO != PRO_NONE && warp >= XF_WARP0 && warp < XF_WARP0 + 4) {
        // ------------------------------------------------------------ transform
        const int t = threadIdx.x - 32 * XF_WARP0;
        const int ni = box_rows / 16;  // rows of this thread: t/8 + 16 i
        float mean[8], rstd[8], ss[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mean[i] = 0.f;
            rstd[i] = 1.f;
            ss[i] = 0.f;
        }
        if (PRO == PRO_LN) {
            const float2* stats = reinterpret_cast<const float2*>(p.ln_stats);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = (t >> 3) + 16 * i;
                if (i < ni && r < rows) {
                    const float2 st = stats[m0 + r];
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
            else if (PRO == PRO_ADD)
                fold_add_stage<DT>(stage_a(s), gb_slot(s), t, ni);
            else
                fold_ln_stage<DT>(stage_a(s), gb_slot(s), p.beta != nullptr, t, ni, mean, rstd);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(xform_bar(s));
            if (++s == NS) {
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
            named_bar_arrive(3, 256);  // hand the partial sums to the epilogue warps
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ reduction exchange + epilogue
        // This tail runs on few warps with little to overlap it, so its
        // index arithmetic comes from host-built tables (no divisions).
        const int q = warp & 3;
        const int r = q * 32 + lane;                 // the row this thread drains
        const int t = threadIdx.x - 32 * EPI_WARP0;  // 0..127
        const int me = rank;
        const int stride = p.xc_stride;              // floats per slot row
        const uint32_t slot_bytes = (uint32_t)(rows * stride) * 4u;
        const uint32_t row_off = (uint32_t)(r * stride) * 4u;
        // slots in the (now idle) ring: [0, splits) received, indexed by
        // sender (my own partial of my slice among them); then splits - 1
        // outgoing, indexed by owner, skipping me
        auto slot_index = [&](int d) { return d == me ? me : splits + d - (d > me ? 1 : 0); };
        const bool lead = t == 0;
        {
            // bring the parameters the tail reads into this SM's constant
            // cache while the main loop runs (a miss there costs an L2
            // round trip on the critical path)
            uint32_t touch = (uint32_t)p.xc_stride ^ p.xc_owner[lane] ^ p.xc_pos[lane] ^ p.xc_c0[lane & 7] ^
                             __float_as_uint(p.inv_k) ^ __float_as_uint(p.eps) ^ (uint32_t)out_act(p, osel.oi) ^
                             (uint32_t)out_n(p, osel.oi) ^ (uint32_t)reinterpret_cast<uintptr_t>(p.residual) ^
                             (uint32_t)reinterpret_cast<uintptr_t>(out_ptr(p, osel.oi)) ^
                             (uint32_t)reinterpret_cast<uintptr_t>(out_bias(p, osel.oi));
            asm volatile("" ::"r"(touch));
        }

        bool ok = wait_bar(tfull_bar, 0, p.status, p.timeout_ns, 24);
        __syncwarp();
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        float ssr = 0.f;
        if (PRO == PRO_RMS) {
            named_bar_sync(3, 256);  // the transform warps have written ssbuf
            if (r < rows) ssr = ssbuf[r];
        }
        if (ok) {
            tc_fence_after();
            if (lead) FL_MARK(p, 5);
            if (lead && splits > 1) mbar_arrive_expect_tx(recvd_bar, (uint32_t)(splits - 1) * slot_bytes);
            if (q * 32 < rows) {
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
                if constexpr (DUAL) {
                    // gate and up of one 32-column group per wait; a chunk's
                    // slot entry is its 8 gate values, then its 8 up values
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t g[32], u[32];
                        tmem_ld_32x32b_x32(taddr + c * 32, g);
                        tmem_ld_32x32b_x32(taddr + BN + c * 32, u);
                        tmem_ld_wait();
                        if (r < rows) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int ch = c * 4 + j;
                                const uint32_t dst = ring + (uint32_t)slot_index(p.xc_owner[ch]) * slot_bytes +
                                                     row_off + (uint32_t)p.xc_pos[ch] * (uint32_t)(C::CHUNK_FLOATS * 4);
                                st_shared_v4(dst, g[j * 8], g[j * 8 + 1], g[j * 8 + 2], g[j * 8 + 3]);
                                st_shared_v4(dst + 16, g[j * 8 + 4], g[j * 8 + 5], g[j * 8 + 6], g[j * 8 + 7]);
                                st_shared_v4(dst + 32, u[j * 8], u[j * 8 + 1], u[j * 8 + 2], u[j * 8 + 3]);
                                st_shared_v4(dst + 48, u[j * 8 + 4], u[j * 8 + 5], u[j * 8 + 6], u[j * 8 + 7]);
                            }
                        }
                    }
                }
                // two 32-column loads in flight per wait
                constexpr int NB = BN / 32 < 2 ? 1 : 2;
#pragma unroll
                for (int c = 0; c < (DUAL ? 0 : BN / 32); c += NB) {
                    uint32_t v[NB][32];
#pragma unroll
                    for (int b = 0; b < NB; ++b) tmem_ld_32x32b_x32(taddr + (c + b) * 32, v[b]);
                    tmem_ld_wait();
                    if (r < rows) {
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int ch = (c + b) * 4 + j;
                                const uint32_t dst = ring + (uint32_t)slot_index(p.xc_owner[ch]) * slot_bytes +
                                                     row_off + (uint32_t)p.xc_pos[ch] * 32u;
                                st_shared_v4(dst, v[b][j * 8], v[b][j * 8 + 1], v[b][j * 8 + 2], v[b][j * 8 + 3]);
                                st_shared_v4(dst + 16, v[b][j * 8 + 4], v[b][j * 8 + 5], v[b][j * 8 + 6],
                                             v[b][j * 8 + 7]);
                            }
                        }
                    }
                }
                if (PRO == PRO_RMS && r < rows) {
                    const uint32_t ss_off = row_off + (uint32_t)(stride - 4) * 4u;
#pragma unroll
                    for (int d = 0; d < 8; ++d)
                        if (d < splits) st_shared_f32(ring + (uint32_t)slot_index(d) * slot_bytes + ss_off, ssr);
                }
            }
            if (lead) FL_MARK(p, 10);
            tc_fence_before();
            fence_proxy_async_smem();  // outgoing slots are read by the bulk copies
            named_bar_sync(2, 128);
            if (lead && splits > 1) {
                if (wait_bar_cluster(peerfree_bar, 0, p.status, p.timeout_ns, 25)) {
                    const uint32_t src0 = ring + (uint32_t)splits * slot_bytes;
                    const uint32_t dst = ring + (uint32_t)me * slot_bytes;
                    for (int d = 0, k = 0; d < splits; ++d) {
                        if (d == me) continue;
                        bulk_copy_to_cluster(mapa_cluster(dst, (uint32_t)d), src0 + (uint32_t)k * slot_bytes, slot_bytes,
                                             mapa_cluster(recvd_bar, (uint32_t)d));
                        ++k;
                    }
                }
                FL_MARK(p, 6);
            }
            if (splits > 1) ok = wait_bar_cluster(recvd_bar, 0, p.status, p.timeout_ns, 26);
            if (lead) FL_MARK(p, 7);
        }
        if (lead) xchg_ok = ok ? 1 : 0;
        __syncwarp();
        // my incoming partials are in, so every peer's copy to me has read
        // its source: the second half of the lifetime barrier can open
        cluster_arrive_relaxed();
        if (lead) FL_MARK(p, 11);
    }

    if (warp < EPI_WARP0) {
        __syncwarp();
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        if (warp == 1 && lane == 0 && ring_idle && splits > 1) {
            // my MMAs are done with my ring: peers may write their partials
            // of my slice into it
            for (int d = 0; d < splits; ++d)
                if (d != rank) mbar_arrive_cluster(mapa_cluster(peerfree_bar, (uint32_t)d));
        }
        __syncwarp();
        cluster_arrive_relaxed();  // nothing below touches another CTA
    }
    // ---------------------------------------------------------------- reduction + epilogue
    // Every thread of the CTA sums the `splits` partials of my slice (rows x
    // w chunks of 8 columns; w rounded up to a power of two threads per row,
    // one chunk each),
    // scales, adds bias, activation and residual, and stores 16 bytes.
    const int xc0 = p.xc_c0[rank];
    const int xw = p.xc_c0[rank + 1] - xc0;
    const int xsh = xw > 1 ? 32 - __clz(xw - 1) : 0;  // 2^xsh >= xw threads per row
    const int xch = threadIdx.x & ((1 << xsh) - 1);
    const int xcol = n0 + (xc0 + xch) * 8;
    const int N = out_n(p, osel.oi);
    const int act = out_act(p, osel.oi);
    const void* obias = out_bias(p, osel.oi);
    const bool xmine = xch < xw && xcol < N;
    float bb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) bb[e] = 0.f;
    if (xmine && obias != nullptr) {  // in flight across the barrier
        const uint4 bv = ldg_v4(reinterpret_cast<const uint16_t*>(obias) + xcol);
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 b2 = Ops::unpack(bw[e]);
            bb[2 * e] = b2.x;
            bb[2 * e + 1] = b2.y;
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // the epilogue warps saw every partial of my slice land
    if (threadIdx.x == 0) FL_MARK(p, 12);
    if (xchg_ok && xmine) {
        using T = uint16_t;
        const T* res = reinterpret_cast<const T*>(p.residual);
        T* out = reinterpret_cast<T*>(out_ptr(p, osel.oi));
        const int stride = p.xc_stride;
        const uint32_t slot_bytes = (uint32_t)(rows * stride) * 4u;
        const int nthreads = (int)blockDim.x;
        for (int row = (int)threadIdx.x >> xsh; row < rows; row += nthreads >> xsh) {
            const size_t g = (size_t)(m0 + row) * N + xcol;
            uint4 rv = make_uint4(0u, 0u, 0u, 0u);
            if (res != nullptr) rv = *reinterpret_cast<const uint4*>(res + g);
            float v[8], vu[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = vu[e] = 0.f;
            float ss = 0.f;
            const uint32_t a0 = ring + (uint32_t)(row * stride + xch * C::CHUNK_FLOATS) * 4u;
            const uint32_t s0 = ring + (uint32_t)(row * stride + stride - 4) * 4u;
#pragma unroll
            for (int src = 0; src < 8; ++src) {
                if (src < splits) {
                    const uint32_t a = a0 + (uint32_t)src * slot_bytes;
                    const uint4 lo = ld_shared_v4(a), hi = ld_shared_v4(a + 16);
                    v[0] += __uint_as_float(lo.x); v[1] += __uint_as_float(lo.y);
                    v[2] += __uint_as_float(lo.z); v[3] += __uint_as_float(lo.w);
                    v[4] += __uint_as_float(hi.x); v[5] += __uint_as_float(hi.y);
                    v[6] += __uint_as_float(hi.z); v[7] += __uint_as_float(hi.w);
                    if (DUAL) {
                        const uint4 ulo = ld_shared_v4(a + 32), uhi = ld_shared_v4(a + 48);
                        vu[0] += __uint_as_float(ulo.x); vu[1] += __uint_as_float(ulo.y);
                        vu[2] += __uint_as_float(ulo.z); vu[3] += __uint_as_float(ulo.w);
                        vu[4] += __uint_as_float(uhi.x); vu[5] += __uint_as_float(uhi.y);
                        vu[6] += __uint_as_float(uhi.z); vu[7] += __uint_as_float(uhi.w);
                    }
                    if (PRO == PRO_RMS) ss += ld_shared_f32(s0 + (uint32_t)src * slot_bytes);
                }
            }
            const float rs = PRO == PRO_RMS ? rsqrtf(fmaf(ss, p.inv_k, p.eps)) : 1.f;
            if (DUAL) {
                // h = silu(gate) * up, both scaled by 1/rms
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = act_apply(ACT_SILU, v[e] * rs) * (vu[e] * rs);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = fmaf(v[e], rs, bb[e]);
            }
            if (!DUAL && act != ACT_NONE) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = act_apply(act, v[e]);
            }
            if (res != nullptr) {
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 r2 = Ops::unpack(rw[e]);
                    v[2 * e] += r2.x;
                    v[2 * e + 1] += r2.y;
                }
            }
            if (threadIdx.x == 0) FL_MARK(p, 13);
            *reinterpret_cast<uint4*>(out + g) = make_uint4(Ops::pack(v[0], v[1]), Ops::pack(v[2], v[3]),
                                                             Ops::pack(v[4], v[5]), Ops::pack(v[6], v[7]));
        }
    }
    if (threadIdx.x == 0) FL_MARK(p, 8);
    __syncwarp();
    // no CTA leaves while a peer may still read or write its shared memory
    cluster_wait();
    if (threadIdx.x == 0) FL_MARK(p, 9);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int DT, int BN, int PRO, bool DUAL, bool MULTI>
cudaError_t splitk_configure() {
    static cudaError_t state = [] {
        auto kern = fl_splitk_kernel<DT, BN, PRO, DUAL, MULTI>;
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SplitCfg<BN, DUAL>::SMEM_MAX);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        return e;
    }();
    return state;
}

// How many clusters of `splits` CTAs of this kernel, each with `smem_bytes`
// of dynamic shared memory, can be resident at once.
template <int DT, int BN, int PRO, bool DUAL>
int splitk_max_clusters(int splits, int smem_bytes) {
    if (splitk_configure<DT, BN, PRO, DUAL, false>() != cudaSuccess) return 0;
    auto kern = fl_splitk_kernel<DT, BN, PRO, DUAL, false>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, 1, 1);
    cfg.blockDim = dim3(splitk_threads<PRO>(), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
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

template <int DT, int BN, int PRO, bool DUAL, bool MULTI>
cudaError_t launch_splitk(const ParamsT<MULTI>& p, int grid, int splits, cudaStream_t stream) {
    using C = SplitCfg<BN, DUAL>;
    auto kern = fl_splitk_kernel<DT, BN, PRO, DUAL, MULTI>;
    cudaError_t e = splitk_configure<DT, BN, PRO, DUAL, MULTI>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(splitk_threads<PRO>(), 1, 1);
    cfg.dynamicSmemBytes = C::smem_bytes(p.s_stages, p.s_stage_bytes);
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
