// CTA-pair fused dense-layer kernel for sm_103a (tcgen05.mma.cta_group::2).
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile per
// step: CTA r stages activation rows [128 r, 128 r + 128) of the tile and
// weight rows [128 r, 128 r + 128) of its 256 columns; the leader (rank 0)
// issues one 256 x 256 x 16 MMA per K slice, whose operands come from both
// shared memories and whose accumulator rows land 128 / 128 in the two tensor
// memories. Each SM therefore stages and reads only half of the weight tile:
// per 64-wide K slice an SM moves 64 KB through shared memory for 512 cycles
// of MMA work (a single-CTA 128 x 256 tile moves 96 KB for the same work).
//
// Plain patterns keep both operands in shared memory and double-buffer the
// accumulator (2 x 256 TMEM columns). Norm prologues fold the activation into
// tensor memory (thread t of the transform warpgroup owns row t), so the MMA
// reads A from TMEM; the accumulator is then single-buffered (256 columns +
// 6 x 32 activation columns; with 128-wide tiles both accumulator buffers
// still fit).
//
// Barriers: `full` (leader) counts the bytes of both CTAs' weight halves (and,
// for plain patterns, of both activation halves) through the pair form of the
// TMA load; `afull` (each CTA) counts that CTA's activation and gamma/beta
// slices for its fold; `xform` (leader) collects the fold warps of both CTAs;
// `empty`, `tfull` are signalled in both CTAs by multicast commits; `tempty`
// (leader) collects both CTAs' epilogue warps. Every wait is bounded.
#pragma once

#include "fl_common.cuh"
#include "fl_fold.cuh"

namespace fl {

template <int BN_, int PRO, int KS = 1>
struct PairCfg {
    static constexpr int BN = BN_;       // output columns of a pair tile (128 or 256)
    static constexpr int HALF = BN / 2;  // weight rows staged per CTA
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = HALF * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr bool ATMEM = PRO != PRO_NONE;  // norm prologues fold into TMEM
    static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = ATMEM ? (STAGES_RAW > 6 ? 6 : STAGES_RAW) : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
    // double-buffer the accumulator unless the activation slots need the room
    // (split-K clusters compute one tile each)
    static constexpr int NBUF = (KS == 2 || (ATMEM && 2 * BN + 32 * STAGES > 512)) ? 1 : 2;
    static constexpr int ACC_COLS = BN;
    static constexpr int A_COL0 = NBUF * ACC_COLS;
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_BUF_BYTES = 32 * 128;
    static constexpr int OFF_EPI = STAGES * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + 4 * EPI_BUF_BYTES;
    // split-K exchange: the K-partner's half of the partial tile, written into
    // this CTA's (idle) ring in 32-column chunks, each as four 32-row blocks
    // (one per epilogue warp, one bulk copy each), so the receiver finishes a
    // chunk while the next is in flight. A block row is 32 fp32 values plus 4
    // words (the first carries the row's partial sum of squares in chunk 0):
    // 36 words keep rows on distinct banks for 16-byte accesses.
    static constexpr int XCOLS = 32;
    static constexpr int NCHUNK = BN / 2 / XCOLS;
    static constexpr int XROW = XCOLS + 4;                      // words per block row
    static constexpr int XBLOCK = 32 * XROW * 4;                // one warp's rows of one chunk
    static constexpr int XCHUNK = 4 * XBLOCK;
    static constexpr int XCHG_BYTES = NCHUNK * XCHUNK;
    static constexpr int OFF_SEND = 96 * 1024;                  // outgoing blocks, same layout
    static constexpr int NUM_BARS = 4 * STAGES + 10 + 4 * NCHUNK;
    static_assert(KS == 1 || OFF_SEND + XCHG_BYTES <= STAGES * STAGE_BYTES, "exchange buffers fit in the ring");
    static_assert(XCHG_BYTES <= OFF_SEND && XCHG_BYTES % 16 == 0, "exchange layout");
    // second set of epilogue staging buffers (split-K: the ring is idle by then)
    static constexpr int OFF_EPI2 = (XCHG_BYTES + 1023) / 1024 * 1024;
    static_assert(KS == 1 || OFF_EPI2 + 4 * EPI_BUF_BYTES <= OFF_SEND, "second staging set fits in the ring");
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ROWSCALE = (OFF_SLOT + 16 + 15) / 16 * 16;
    static constexpr int OFF_GB = (OFF_ROWSCALE + 2 * kBM * 4 + 127) / 128 * 128;
    // each epilogue warp's copy of the tile's bias slice (BN x 16-bit)
    static constexpr int OFF_BIAS = OFF_GB + STAGES * 256;
    static constexpr int SMEM_BYTES = OFF_BIAS + 4 * BN * 2 + 1024;
    static_assert(!ATMEM || A_COL0 + 32 * STAGES <= TMEM_COLS, "activation slots must fit in tensor memory");
};

// DUAL (SwiGLU gate/up): the 256-row weight tile of a pair is rows
// [n0, n0 + 128) of Wg (even CTA) stacked over the same rows of Wu (odd CTA),
// so one 256 x 256 MMA yields gate | up for 128 output columns, and the
// epilogue writes silu(gate) * up.
template <int DT, int BN, int PRO, int KS, bool DUAL, bool MULTI>
__global__ void __launch_bounds__(PRO != PRO_NONE ? 384 : 256, 1)
    fl_pair_kernel(const __grid_constant__ ParamsT<MULTI> p) {
    using C = PairCfg<BN, PRO, KS>;
    static_assert(!DUAL || (BN == 256 && KS == 1), "gate/up pairs use 256-wide tiles without a K split");
    constexpr int OUT_COLS = DUAL ? BN / 2 : BN;  // output columns of a tile
    static_assert(KS == 1 || (KS == 2 && BN == 256), "split-K pairs use 256-wide tiles");
    if (threadIdx.x == 0) FL_MARK(p, 0);
    using Ops = DTypeOps<DT>;
    constexpr int S = C::STAGES;
    constexpr int EPI_WARP0 = PRO != PRO_NONE ? 8 : 4;
    // fp16 LayerNorm with a single accumulator buffer: the epilogue warps, idle
    // while a tile's MMAs run, take a share of the fold. SHARE_ALT: the fold
    // warps fold whole rows of the even K blocks (by a running block index)
    // and the epilogue warps those of the odd ones, so each warpgroup has two
    // MMA steps for one fold; SHARE_SPLIT: the fold warps fold chunks 0-3 of
    // every K block and the epilogue warps chunks 4-7. The RMSNorm and
    // input-bias folds keep pace with the MMAs on the fold warps alone and
    // measured faster unshared (the bench default 17.6 against 18.0 us,
    // rmsnorm_gemm 4096^3 102.1 against 103.7 us); LayerNorm fp16 at 4096^3
    // took 134.5 us unshared against 127.3 alternating, but LayerNorm bf16
    // (whose fold widens with one mixed-precision FMA) 126.4 against 131.7,
    // so only fp16 LayerNorm shares.
    constexpr int SHARE_NONE = 0, SHARE_SPLIT = 1, SHARE_ALT = 2;
#ifndef FL_PAIR_SHARE
#define FL_PAIR_SHARE 2
#endif
    constexpr int SHARE = (PRO == PRO_LN && DT == DT_F16 && C::NBUF == 1) ? FL_PAIR_SHARE : SHARE_NONE;
    constexpr bool FOLD2 = SHARE != SHARE_NONE;
    static_assert(SHARE != SHARE_ALT || S % 2 == 0, "alternating folds need an even ring: a warpgroup's "
                  "blocks k and k + S must share a stage's phase sequence");
    constexpr uint32_t IDESC = umma_idesc_f16(Ops::kFormat, 2 * kBM, C::BN);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw_addr);

    auto stage_a = [&](int s) { return sbase + s * C::STAGE_BYTES; };
    auto stage_b = [&](int s) { return sbase + s * C::STAGE_BYTES + C::A_BYTES; };
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto afull_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    // (norm prologues: the folds of both CTAs arrive on the leader's `full`
    // barrier itself, so the MMA thread tests one barrier per K step)
    auto xform_bar = [&](int s) { return bar0 + 8u * s; };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (4 * S + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (4 * S + 2 + b); };
    auto sready_bar = [&](int b) { return bar0 + 8u * (4 * S + 4 + b); };
    const uint32_t drain_bar = bar0 + 8u * (4 * S + 6);
    const uint32_t tdone_bar = bar0 + 8u * (4 * S + 7);  // this CTA's epilogue finished a tile
    const uint32_t ringfree_bar = bar0 + 8u * (4 * S + 8);  // split-K: the K-partner may write my ring
    // split-K: block (warp q, chunk c) of the K-partner's half has arrived
    auto recvd_bar = [&](int q, int c) { return bar0 + 8u * (4 * S + 10 + q * C::NCHUNK + c); };
    const uint32_t slot_addr = sbase + C::OFF_SLOT;
    float* rowscale = reinterpret_cast<float*>(smem + C::OFF_ROWSCALE);
    auto gb_slot = [&](int s) { return sbase + C::OFF_GB + 256u * s; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Cluster of 2 (one pair) or, with KS = 2, of 4: two pairs, one per K half
    // of the same tile. Pair peers differ in rank bit 0; the leader is even.
    const uint32_t crank = cluster_rank();
    const uint32_t rank = crank & 1u;
    const uint32_t lead_rank = crank & ~1u;
    const bool leader = rank == 0;
    const uint16_t pair_mask = (uint16_t)(0x3u << lead_rank);
    auto lead = [&](uint32_t local_addr) { return mapa_cluster(local_addr, lead_rank); };  // leader's copy
    const int nk = p.num_k_blocks;
    const int khalf = KS == 2 ? (int)(crank >> 1) : 0;
    const int kb_begin = KS == 2 ? khalf * p.kps : 0;
    const int kb_end = KS == 2 ? min(nk, kb_begin + p.kps) : nk;
    // KS = 1: persistent pairs take the tiles round-robin (pair q: q,
    // q + npairs, ...), so the tiles in flight form a compact band and the
    // operand they share is read from HBM once. Row-block-major for one
    // weight (a band of row blocks over every column block: the weight stays
    // hot in L2 while the activation rows stream through once; contiguous
    // ranges per pair spread the tiles in flight over the whole grid and
    // re-read the weight from HBM: gemm_bias at 4096^3 2.4 % slower).
    // Column-block-major for the gate/up pair, whose Wg + Wu (180 MB at
    // F = 11008) do not fit in L2 while the activation does: a band of column
    // blocks over every row block, each weight tile read from HBM once
    // (contiguous ranges had re-read it for every row block: 2.4 GB of DRAM
    // reads per 4096-row launch against 0.2 GB of operands). KS = 2: one tile
    // per cluster.
    const int npairs = KS == 2 ? p.num_tiles : (int)gridDim.x / 2;
    const int pair = KS == 2 ? (int)blockIdx.x / 4 : (int)blockIdx.x / 2;
    int t_begin = pair, t_end = pair + 1, t_step = 1;
    if (KS == 1) {
        t_end = p.num_tiles;
        t_step = npairs;
    }
    auto tile_mb = [&](int t) { return DUAL ? t % p.num_m_blocks : t / p.num_n_blocks; };
    auto tile_nb = [&](int t) { return DUAL ? t / p.num_m_blocks : t % p.num_n_blocks; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), PRO != PRO_NONE ? 1 + (SHARE == SHARE_SPLIT ? 16 : 8) : 1);
            mbar_init(afull_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 8);
            mbar_init(sready_bar(b), 4);
        }
        mbar_init(drain_bar, 1);
        mbar_init(tdone_bar, 4);
        mbar_init(ringfree_bar, 4);
        for (int i = 0; i < 4 * C::NCHUNK; ++i) mbar_init(recvd_bar(i / C::NCHUNK, i % C::NCHUNK), 1);
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
        tmem_alloc_pair(slot_addr, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_barrier_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);
    // L2 prefetch of this CTA's first weight tiles overlaps the previous kernel
    // (L2 is the point of coherence); every other global access waits for it.
    // (Issuing it, with the activation tiles, before the set-up above made
    // the set-up slower than the prefetch saved: 19.4 against 18.8 us at
    // 512 x 4096 x 4096.)
    if (warp == 0 && lane == 0 && t_begin < t_end) {
        const OutSel o = out_sel(p, tile_nb(t_begin));
        const int nh = DUAL ? o.nb * OUT_COLS : o.nb * C::BN + (int)rank * C::HALF;
        const CUtensorMap* tb = DUAL && rank ? &p.tmB2 : tm_b(p, o.oi);
        for (int kb = kb_begin; kb < kb_begin + S && kb < kb_end; ++kb) tma_prefetch_2d(tb, kb * kBK, nh);
    }
    // LayerNorm: this grid directly follows the row-statistics kernel, which
    // lets dependents launch only after its own dependency wait, so every
    // kernel before it has completed and every input but the statistics is
    // final when this grid starts. Only the warps that read the statistics
    // (fold, and with the split fold epilogue, warps) wait for it; the
    // producer fills the ring meanwhile.
    constexpr int kTrigger = PRO == PRO_LN ? 128 : 0;
    if (PRO != PRO_LN || warp >= 4) griddep_wait();
    if (threadIdx.x == kTrigger) griddep_launch_dependents();
    if (threadIdx.x == 0) FL_MARK(p, 1);

    // The bias of tile columns [n0, n0 + BN) into this epilogue warp's own
    // shared buffer (one 16-byte load per lane and 256 columns; zeros past N),
    // before the accumulator is waited for: the epilogue then reads it with
    // broadcast shared loads instead of global loads on its critical path.
    auto stage_bias = [&](int n0, int q, int oi) -> uint32_t {
        const uint32_t buf = sbase + C::OFF_BIAS + (uint32_t)(q * C::BN * 2);
        if (out_bias(p, oi) != nullptr) {
            const uint16_t* b = reinterpret_cast<const uint16_t*>(out_bias(p, oi));
            for (int c = (int)(threadIdx.x & 31) * 8; c < C::BN; c += 256) {
                const uint4 v = n0 + c < out_n(p, oi) ? ldg_v4(b + n0 + c) : make_uint4(0u, 0u, 0u, 0u);
                st_shared_v4(buf + (uint32_t)c * 2u, v.x, v.y, v.z, v.w);
            }
        }
        __syncwarp();
        return buf;
    };

    // One tile's fold of chunks [j0, j0 + 4) of every K block of row rl into
    // the lower (j0 = 0) or upper (j0 = 4) 16 columns of the stage's TMEM slot
    // (FOLD2: the fold warps take chunks 0-3, the epilogue warps 4-7). The
    // loads of block kb + 1 go into the other register set once block kb has
    // been handed to the MMA: issuing them before block kb's TMEM store, to
    // overlap their latency with its arithmetic, was measured 15 % slower (the
    // store, and with it the hand-off, then waits behind them). (fs, fph): ring
    // position, kept by the caller across tiles; ssum: RMS sum of squares of
    // the row over these chunks.
    //
    // SHARE_ALT (fold_share below): warpgroup wg folds whole rows of the K
    // blocks whose running index g (counted over every block of every tile,
    // the same in both warpgroups) has parity wg, and only advances its ring
    // position over the others.
    auto fold_tile = [&](int tile, int rl, int j0, int& fs, uint32_t& fph, float& ssum, int site) -> bool {
        float rstd = 1.f, nmr = 0.f;
        if (PRO == PRO_LN) {
            const int row = tile_mb(tile) * 2 * kBM + (int)rank * kBM + rl;
            if (row < p.M) {
                const float2 st = reinterpret_cast<const float2*>(p.ln_stats)[row];
                rstd = st.y;
                nmr = -st.x * st.y;
            }
        }
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t a_cols = tmem_base + ((uint32_t)(rl & ~31) << 16) + (uint32_t)C::A_COL0 + 4u * (uint32_t)j0;
        const bool has_beta = p.beta != nullptr;
        using R = FoldRegs<4, PRO == PRO_LN>;
        R ra, rb;
        if (!wait_bar(afull_bar(fs), fph, p.status, p.timeout_ns, site)) return false;
        fold_row_load(ra, stage_a(fs), gb_slot(fs), has_beta, rl, j0);
        // one K block: fold `cur` (ring position fs), then load the next into `nxt`
        auto step = [&](R& cur, R& nxt, bool has_next) -> bool {
            uint32_t o[16];
            if constexpr (PRO == PRO_LN)
                fold_ln_compute<DT>(cur, rstd, nmr, o);
            else if constexpr (PRO == PRO_ADD)
                fold_add_compute<DT>(cur, o);
            else
                fold_rms_compute<DT>(cur, ss, o);
            tmem_st_32x32b_x16(a_cols + 32u * (uint32_t)fs, o);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lead(xform_bar(fs)));
            if (++fs == S) {
                fs = 0;
                fph ^= 1u;
            }
            if (has_next) {
                if (!wait_bar(afull_bar(fs), fph, p.status, p.timeout_ns, site)) return false;
                fold_row_load(nxt, stage_a(fs), gb_slot(fs), has_beta, rl, j0);
            }
            return true;
        };
        for (int kb = kb_begin; kb < kb_end; kb += 2) {
            if (!step(ra, rb, kb + 1 < kb_end)) return false;
            if (kb + 1 >= kb_end) break;
            if (!step(rb, ra, kb + 2 < kb_end)) return false;
        }
        ssum = (ss[0] + ss[1]) + (ss[2] + ss[3]);
        return true;
    };

    auto fold_alt = [&](int tile, int rl, int wg, int& fs, uint32_t& fph, int& g, float& ssum, int site) -> bool {
        float rstd = 1.f, nmr = 0.f;
        if (PRO == PRO_LN) {
            const int row = tile_mb(tile) * 2 * kBM + (int)rank * kBM + rl;
            if (row < p.M) {
                const float2 st = reinterpret_cast<const float2*>(p.ln_stats)[row];
                rstd = st.y;
                nmr = -st.x * st.y;
            }
        }
        float ss[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ss[i] = 0.f;
        const uint32_t a_cols = tmem_base + ((uint32_t)(rl & ~31) << 16) + (uint32_t)C::A_COL0;
        const bool has_beta = p.beta != nullptr;
        for (int kb = kb_begin; kb < kb_end; ++kb, ++g) {
            if ((g & 1) == wg) {
                if (!wait_bar(afull_bar(fs), fph, p.status, p.timeout_ns, site)) return false;
                if (rl == 0 && tile == t_begin) FL_MARK_STEP(p, 24, kb - kb_begin);
                uint32_t o[32];
                if (PRO == PRO_RMS) {
                    fold_rms_row<DT>(stage_a(fs), gb_slot(fs), rl, ss, o);
                } else if (PRO == PRO_ADD) {
                    fold_add_row<DT>(stage_a(fs), gb_slot(fs), rl, o);
                } else {
                    uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[0]);
                    uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(&o[16]);
                    fold_ln_row<DT, 4, 0>(stage_a(fs), gb_slot(fs), has_beta, rl, rstd, nmr, lo);
                    fold_ln_row<DT, 4, 4>(stage_a(fs), gb_slot(fs), has_beta, rl, rstd, nmr, hi);
                }
                tmem_st_32x32b_x32(a_cols + 32u * (uint32_t)fs, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(lead(xform_bar(fs)));
                if (rl == 0 && tile == t_begin) FL_MARK_STEP(p, 32, kb - kb_begin);
            }
            if (++fs == S) {
                fs = 0;
                fph ^= 1u;
            }
        }
        ssum = ((ss[0] + ss[1]) + (ss[2] + ss[3])) + ((ss[4] + ss[5]) + (ss[6] + ss[7]));
        return true;
    };

    // This warpgroup's share of a tile's fold (wg 0: fold warps, 1: epilogue warps).
    auto fold_share = [&](int tile, int rl, int wg, int& fs, uint32_t& fph, int& g, float& ssum, int site) -> bool {
        if constexpr (SHARE == SHARE_ALT) return fold_alt(tile, rl, wg, fs, fph, g, ssum, site);
        return fold_tile(tile, rl, 4 * wg, fs, fph, ssum, site);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            const uint32_t gb_bytes = PRO != PRO_NONE ? 128u + (PRO == PRO_LN && p.beta != nullptr ? 128u : 0u) : 0u;
            for (int tile = t_begin; ok && tile < t_end; tile += t_step) {
                const int m0 = tile_mb(tile) * 2 * kBM + (int)rank * kBM;
                // this CTA's weight rows: its half of the tile, or (DUAL) the
                // tile's rows of Wg / Wu
                const OutSel o = out_sel(p, tile_nb(tile));
                const int nh = DUAL ? o.nb * OUT_COLS : o.nb * C::BN + (int)rank * C::HALF;
                const CUtensorMap* tb = DUAL && rank ? &p.tmB2 : tm_b(p, o.oi);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bar(empty_bar(s), ph ^ 1u, p.status, p.timeout_ns, 31)) {
                        ok = false;
                        break;
                    }
                    if (tile == t_begin) FL_MARK_STEP(p, 16, kb - kb_begin);
                    if (PRO == PRO_NONE) {
                        if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * C::STAGE_BYTES);
                        const uint32_t fb = lead(full_bar(s));
                        tma_load_2d_pair(stage_a(s), &p.tmA, fb, kb * kBK, m0);
                        tma_load_2d_pair(stage_b(s), tb, fb, kb * kBK, nh);
                    } else {
                        mbar_arrive_expect_tx(afull_bar(s), (uint32_t)C::A_BYTES + gb_bytes);
                        tma_load_2d(stage_a(s), &p.tmA, afull_bar(s), kb * kBK, m0);
                        tma_load_2d(gb_slot(s), &p.tmGamma, afull_bar(s), kb * kBK, 0);
                        if (PRO == PRO_LN && p.beta != nullptr)
                            tma_load_2d(gb_slot(s) + 128, &p.tmBeta, afull_bar(s), kb * kBK, 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(s), 2u * C::B_BYTES);
                        tma_load_2d_pair(stage_b(s), tb, lead(full_bar(s)), kb * kBK, nh);
                    }
                    if (issued == 0) FL_MARK(p, 2);
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Drain: the leader's `full` covers both CTAs' pair loads; each CTA's
            // `afull` covers its own activation loads.
            const int pending = issued < S ? issued : S;
            for (int i = 1; i <= pending; ++i) {
                const int idx = issued - i;
                const uint32_t par = (uint32_t)((idx / S) & 1);
                if (leader) wait_bar_drain(full_bar(idx % S), par, 20000000ull);
                if (PRO != PRO_NONE) wait_bar_drain(afull_bar(idx % S), par, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int tile = t_begin; ok && tile < t_end; tile += t_step, ++it) {
                const int buf = C::NBUF == 2 ? (it & 1) : 0;
                const uint32_t tph = C::NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
                if (!wait_bar_cluster(tempty_bar(buf), tph ^ 1u, p.status, p.timeout_ns, 34)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * C::ACC_COLS);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (it == 0) FL_MARK_STEP(p, 40, kb - kb_begin);
                    if (!wait_bar_cluster(full_bar(s), ph, p.status, p.timeout_ns, 35)) {
                        ok = false;
                        break;
                    }
                    if (it == 0) FL_MARK_STEP(p, 48, kb - kb_begin);
                    if (it == 0) FL_MARK_STEP(p, 56, kb - kb_begin);
                    tc_fence_after();
                    if (kb == kb_begin && it == 0) FL_MARK(p, 3);
                    const uint64_t da = sw128_kmajor_desc(stage_a(s));
                    const uint64_t db = sw128_kmajor_desc(stage_b(s));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t acc = (kb != kb_begin) || (kk != 0);
                        if (C::ATMEM)
                            umma_f16_ts_pair(d, tmem_base + (uint32_t)C::A_COL0 + 32u * s + 8u * kk, db + 2 * kk, IDESC,
                                             acc);
                        else
                            umma_f16_ss_pair(d, da + 2 * kk, db + 2 * kk, IDESC, acc);
                    }
                    umma_commit_pair(empty_bar(s), pair_mask);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(tfull_bar(buf), pair_mask);
                FL_MARK(p, 4);
            }
            umma_commit_pair(drain_bar, (uint16_t)(1u << lead_rank));
            wait_bar_drain(drain_bar, 0, 20000000ull);
        }
    } else if (PRO != PRO_NONE && warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ fold into TMEM (both CTAs)
        const int t = threadIdx.x - 128;
        const uint32_t a_lane = (uint32_t)(32 * (warp & 3)) << 16;
        int s = 0;
        uint32_t ph = 0;
        int it = 0;
        int g = 0;  // running K-block index (SHARE_ALT)
        bool ok = true;
        for (int tile = t_begin; ok && tile < t_end; tile += t_step, ++it) {
            float ssum = 0.f;  // RMS: the row's sum of squares over the blocks / chunks folded here
            if (FOLD2) {
                ok = fold_share(tile, t, 0, s, ph, g, ssum, 38);
            } else {
                float ss[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ss[i] = 0.f;
                float rstd = 1.f, nmr = 0.f;  // LayerNorm: 1/std and -mean/std of row t of this tile
                if (PRO == PRO_LN) {
                    const int row = tile_mb(tile) * 2 * kBM + (int)rank * kBM + t;
                    if (row < p.M) {
                        const float2 st = reinterpret_cast<const float2*>(p.ln_stats)[row];
                        rstd = st.y;
                        nmr = -st.x * st.y;
                    }
                }
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bar(afull_bar(s), ph, p.status, p.timeout_ns, 38)) {
                        ok = false;
                        break;
                    }
                    if (t == 0 && it == 0) FL_MARK_STEP(p, 24, kb - kb_begin);
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
                    if (t == 0 && kb == kb_begin && it == 0) FL_MARK(p, 10);
                    tmem_st_32x32b_x32(tmem_base + a_lane + (uint32_t)C::A_COL0 + 32u * s, o);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(lead(xform_bar(s)));
                    if (t == 0 && it == 0) FL_MARK_STEP(p, 32, kb - kb_begin);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                ssum = ((ss[0] + ss[1]) + (ss[2] + ss[3])) + ((ss[4] + ss[5]) + (ss[6] + ss[7]));
            }
            if (!ok) break;
            if (PRO == PRO_RMS) {
                // row scales of tile `it` go to buffer it & 1; this CTA's epilogue of
                // tile it - 2 (same buffer) has read it once it has finished tile it - 1
                const int rb = it & 1;
                const uint32_t tph = (uint32_t)(it & 1);
                if (!wait_bar(tdone_bar, tph ^ 1u, p.status, p.timeout_ns, 39)) break;
                // split-K or split fold: the raw partial sum, which the epilogue
                // completes (the K-partner's, the upper chunks')
                rowscale[rb * kBM + t] = (KS == 2 || FOLD2) ? ssum : rsqrtf(ssum / (float)p.K + p.eps);
                __syncwarp();
                if (lane == 0) mbar_arrive(sready_bar(rb));
            }
        }
    } else if (KS == 2 && warp >= EPI_WARP0) {
        // ------------------------------------------------------------ split-K epilogue
        // Each CTA owns half of the tile's columns (its K half's index); it ships
        // the other half of its fp32 partial to the K-partner (same rows, other
        // K half) and adds the partner's share of its own half.
        const int q = warp & 3;
        const int rl = q * 32 + lane;  // tile row = TMEM lane
        const uint32_t ebuf = sbase + C::OFF_EPI + q * C::EPI_BUF_BYTES;
        const int sw = lane & 7;
        const uint32_t partner = crank ^ 2u;
        constexpr int HALF_N = C::BN / 2;
        const int tile = pair;
        const int m0 = tile_mb(tile) * 2 * kBM + (int)rank * kBM;
        const OutSel osel = out_sel(p, tile_nb(tile));
        const int n0 = osel.nb * C::BN;
        const int N = out_n(p, osel.oi);
        const int act = out_act(p, osel.oi);
        const int own_c0 = khalf * HALF_N, oth_c0 = (1 - khalf) * HALF_N;
        const uint32_t bias_s = stage_bias(n0, q, osel.oi);
        const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t row_off = (uint32_t)(rl * C::XROW) * 4u;  // within a chunk
        using T = uint16_t;
        const T* bias = reinterpret_cast<const T*>(out_bias(p, osel.oi));
        const T* res = reinterpret_cast<const T*>(p.residual);
        bool ok = true;
        float ss_upper = 0.f;  // RMS, shared fold: the row's sum of squares over this warpgroup's share
        if (FOLD2) {
            int fs = 0, g = 0;
            uint32_t fph = 0;
            ok = fold_share(tile, rl, 1, fs, fph, g, ss_upper, 47);
        }
        ok = ok && wait_bar(tfull_bar(0), 0, p.status, p.timeout_ns, 42);
        tc_fence_after();
        if (threadIdx.x == 32 * EPI_WARP0) FL_MARK(p, 5);
        float ss_own = 0.f;
        if (ok && PRO == PRO_RMS) {
            ok = wait_bar(sready_bar(0), 0, p.status, p.timeout_ns, 43);
            if (ok) ss_own = rowscale[rl] + ss_upper;
        }
        // this pair's MMAs are done, so this CTA's ring may take the partner's half
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_cluster(mapa_cluster(ringfree_bar, partner));
            for (int c = 0; c < C::NCHUNK; ++c) mbar_arrive_expect_tx(recvd_bar(q, c), (uint32_t)C::XBLOCK);
        }
        // ship the outgoing half chunk by chunk: each warp stages its rows and
        // sends them with one bulk copy as soon as the partner's ring is free
        bool peer_ready = false;
        // (two chunks' tensor-memory loads in flight per wait)
        static_assert(C::NCHUNK % 2 == 0, "chunks are shipped in pairs");
#pragma unroll 1
        for (int c2 = 0; c2 < C::NCHUNK; c2 += 2) {
            uint32_t v[2][32];
            if (ok) {
                tmem_ld_32x32b_x32(tl + (uint32_t)(oth_c0 + C::XCOLS * c2), v[0]);
                tmem_ld_32x32b_x32(tl + (uint32_t)(oth_c0 + C::XCOLS * (c2 + 1)), v[1]);
                tmem_ld_wait();
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = c2 + e;
                const uint32_t blk = (uint32_t)(c * C::XCHUNK + q * C::XBLOCK);
                if (ok) {
                    const uint32_t src_row = sbase + C::OFF_SEND + (uint32_t)(c * C::XCHUNK) + row_off;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(src_row + (uint32_t)(4 * j) * 4u, v[e][4 * j], v[e][4 * j + 1], v[e][4 * j + 2],
                                     v[e][4 * j + 3]);
                    if (PRO == PRO_RMS && c == 0) st_shared_f32(src_row + (uint32_t)C::XCOLS * 4u, ss_own);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (ok && lane == 0) {
                    if (!peer_ready) peer_ready = wait_bar_cluster(ringfree_bar, 0, p.status, p.timeout_ns, 44);
                    if (peer_ready)
                        bulk_copy_to_cluster(mapa_cluster(sbase + blk, partner), sbase + C::OFF_SEND + blk,
                                             (uint32_t)C::XBLOCK, mapa_cluster(recvd_bar(q, c), partner));
                }
            }
        }
        if (threadIdx.x == 32 * EPI_WARP0) FL_MARK(p, 6);
        if (ok) {
            float rs = 1.f;
            const int row = m0 + rl;
            const bool row_ok = row < p.M;
            if (m0 + q * 32 < p.M) {
                for (int c = 0; c < HALF_N / 64; ++c) {
                    const int col0 = n0 + own_c0 + c * 64;
                    if (col0 >= N) break;
                    // the two 64-column chunks use two staging buffers
                    const uint32_t sbuf = c == 0 ? ebuf : sbase + C::OFF_EPI2 + q * C::EPI_BUF_BYTES;
                    const uint32_t srow = sbuf + lane * 128;
                    // both 32-column halves of this CTA's accumulator, one wait
                    uint32_t accp[2][32];
                    tmem_ld_32x32b_x32(tl + (uint32_t)(own_c0 + c * 64), accp[0]);
                    tmem_ld_32x32b_x32(tl + (uint32_t)(own_c0 + c * 64 + 32), accp[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int cbase = col0 + h * 32;
                        const int xc = c * 2 + h;        // exchange chunk
                        const uint32_t recv_row = sbase + (uint32_t)(xc * C::XCHUNK) + row_off;
                        // residual of these 32 columns, requested before the waits
                        // and TMEM loads below so its latency overlaps them
                        uint4 rres[4];
                        if (res != nullptr && row_ok) {
                            const T* rrow = res + (size_t)row * N;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                rres[j] = cbase + j * 8 < N ? *reinterpret_cast<const uint4*>(rrow + cbase + j * 8)
                                                            : make_uint4(0u, 0u, 0u, 0u);
                        }
                        if (!wait_bar_cluster(recvd_bar(q, xc), 0, p.status, p.timeout_ns, 45)) ok = false;
                        if (PRO == PRO_RMS && xc == 0) {
                            const float ss = ss_own + ld_shared_f32(recv_row + (uint32_t)C::XCOLS * 4u);
                            rs = rsqrtf(fmaf(ss, 1.0f / (float)p.K, p.eps));
                        }
                        const uint32_t (&acc)[32] = accp[h];
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 r4 = ld_shared_v4(recv_row + (uint32_t)(4 * j) * 4u);
                            v[4 * j + 0] = (__uint_as_float(acc[4 * j + 0]) + __uint_as_float(r4.x)) * rs;
                            v[4 * j + 1] = (__uint_as_float(acc[4 * j + 1]) + __uint_as_float(r4.y)) * rs;
                            v[4 * j + 2] = (__uint_as_float(acc[4 * j + 2]) + __uint_as_float(r4.z)) * rs;
                            v[4 * j + 3] = (__uint_as_float(acc[4 * j + 3]) + __uint_as_float(r4.w)) * rs;
                        }
                        if (bias != nullptr) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (cbase + j * 8 < N) {
                                    const uint4 bv = ld_shared_v4(bias_s + (uint32_t)(cbase + j * 8 - n0) * 2u);
                                    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 b2 = Ops::unpack(bw[e]);
                                        v[j * 8 + 2 * e] += b2.x;
                                        v[j * 8 + 2 * e + 1] += b2.y;
                                    }
                                }
                            }
                        }
                        if (act != ACT_NONE) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = act_apply(act, v[e]);
                        }
                        if (res != nullptr && row_ok) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (cbase + j * 8 < N) {
                                    const uint32_t rw[4] = {rres[j].x, rres[j].y, rres[j].z, rres[j].w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 r2 = Ops::unpack(rw[e]);
                                        v[j * 8 + 2 * e] += r2.x;
                                        v[j * 8 + 2 * e + 1] += r2.y;
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int chunk = h * 4 + j;
                            st_shared_v4(srow + ((chunk ^ sw) << 4), Ops::pack(v[j * 8 + 0], v[j * 8 + 1]),
                                         Ops::pack(v[j * 8 + 2], v[j * 8 + 3]), Ops::pack(v[j * 8 + 4], v[j * 8 + 5]),
                                         Ops::pack(v[j * 8 + 6], v[j * 8 + 7]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tm_out(p, osel.oi), sbuf, col0, m0 + q * 32);
                        bulk_commit_group();
                    }
                }
            }
        }
        if (threadIdx.x == 32 * EPI_WARP0) FL_MARK(p, 13);
        // every block of the partner's has landed (tiles cut by N skip chunks)
        // before this CTA may reach the exit barrier
        if (ok)
            for (int c = 0; c < C::NCHUNK; ++c) wait_bar_cluster(recvd_bar(q, c), 0, p.status, p.timeout_ns, 46);
        if (lane == 0) bulk_wait_group_read<0>();  // global writes complete with the grid
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const uint32_t ebuf = sbase + C::OFF_EPI + q * C::EPI_BUF_BYTES;
        const uint32_t my_row_addr = ebuf + lane * 128;
        const int sw = lane & 7;
        int it = 0;
        int fs = 0;  // ring position and running K-block index of the fold share
        int g = 0;
        uint32_t fph = 0;
        using T = uint16_t;
        const T* res = reinterpret_cast<const T*>(p.residual);
        for (int tile = t_begin; tile < t_end; tile += t_step, ++it) {
            const int m0 = tile_mb(tile) * 2 * kBM + (int)rank * kBM;
            const OutSel osel = out_sel(p, tile_nb(tile));
            const int n0 = osel.nb * OUT_COLS;
            const int N = out_n(p, osel.oi);
            const int act = out_act(p, osel.oi);
            const T* bias = reinterpret_cast<const T*>(out_bias(p, osel.oi));
            const int buf = C::NBUF == 2 ? (it & 1) : 0;
            const uint32_t tph = C::NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
            const uint32_t bias_s = stage_bias(n0, q, osel.oi);
            float ss_upper = 0.f;  // RMS, shared fold: the row's sum of squares over this warpgroup's share
            if (FOLD2 && !fold_share(tile, q * 32 + lane, 1, fs, fph, g, ss_upper, 47)) break;
            if (!wait_bar(tfull_bar(buf), tph, p.status, p.timeout_ns, 40)) break;
            tc_fence_after();
            float rs = 1.f;
            if (PRO == PRO_RMS) {
                if (!wait_bar(sready_bar(it & 1), (uint32_t)((it >> 1) & 1), p.status, p.timeout_ns, 41)) break;
                rs = rowscale[(it & 1) * kBM + q * 32 + lane];
                if (FOLD2) rs = rsqrtf((rs + ss_upper) / (float)p.K + p.eps);
            }
            const int row = m0 + q * 32 + lane;
            const bool row_ok = row < p.M;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::ACC_COLS);
            // 64-column chunks this warp stores (rows or columns past the
            // output are skipped); the accumulator goes back to the MMA right
            // after the last chunk's TMEM load
            int nchunks = 0;
            if (m0 + q * 32 < p.M)
                while (nchunks < OUT_COLS / 64 && n0 + nchunks * 64 < N) ++nchunks;
            bool released = false;
            auto release_acc = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_cluster(lead(tempty_bar(buf)));
                    mbar_arrive(tdone_bar);
                }
                released = true;
            };
            {
                for (int c = 0; c < nchunks; ++c) {
                    const int col0 = n0 + c * 64;
                    // (one wait for both halves' accumulator columns)
                    uint32_t accp[DUAL ? 1 : 2][32];
                    if (!DUAL) {
                        tmem_ld_32x32b_x32(tbase + c * 64, accp[0]);
                        tmem_ld_32x32b_x32(tbase + c * 64 + 32, accp[DUAL ? 0 : 1]);
                        tmem_ld_wait();
                        if (c == nchunks - 1) release_acc();
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int cbase = col0 + h * 32;
                        // residual of these 32 columns, requested before the waits
                        // and TMEM loads below so its latency overlaps them
                        uint4 rres[4];
                        if (res != nullptr && row_ok) {
                            const T* rrow = res + (size_t)row * N;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                rres[j] = cbase + j * 8 < N ? *reinterpret_cast<const uint4*>(rrow + cbase + j * 8)
                                                            : make_uint4(0u, 0u, 0u, 0u);
                        }
                        float v[32];
                        if (DUAL) {
                            uint32_t acc[32];
                            tmem_ld_32x32b_x32(tbase + c * 64 + h * 32, acc);
                            // gate in accumulator columns [0, 128), up in [128, 256)
                            uint32_t up[32];
                            tmem_ld_32x32b_x32(tbase + OUT_COLS + c * 64 + h * 32, up);
                            tmem_ld_wait();
                            if (h == 1 && c == nchunks - 1) release_acc();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                v[e] = act_apply(ACT_SILU, __uint_as_float(acc[e]) * rs) * (__uint_as_float(up[e]) * rs);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(accp[DUAL ? 0 : h][e]) * rs;
                        }
                        if (!DUAL && bias != nullptr) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (cbase + j * 8 < N) {
                                    const uint4 bv = ld_shared_v4(bias_s + (uint32_t)(cbase + j * 8 - n0) * 2u);
                                    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 b2 = Ops::unpack(bw[e]);
                                        v[j * 8 + 2 * e] += b2.x;
                                        v[j * 8 + 2 * e + 1] += b2.y;
                                    }
                                }
                            }
                        }
                        if (!DUAL && act != ACT_NONE) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = act_apply(act, v[e]);
                        }
                        if (!DUAL && res != nullptr && row_ok) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (cbase + j * 8 < N) {
                                    const uint32_t rw[4] = {rres[j].x, rres[j].y, rres[j].z, rres[j].w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 r2 = Ops::unpack(rw[e]);
                                        v[j * 8 + 2 * e] += r2.x;
                                        v[j * 8 + 2 * e + 1] += r2.y;
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
                            const int chunk = h * 4 + j;
                            st_shared_v4(my_row_addr + ((chunk ^ sw) << 4), Ops::pack(v[j * 8 + 0], v[j * 8 + 1]),
                                         Ops::pack(v[j * 8 + 2], v[j * 8 + 3]), Ops::pack(v[j * 8 + 4], v[j * 8 + 5]),
                                         Ops::pack(v[j * 8 + 6], v[j * 8 + 7]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tm_out(p, osel.oi), ebuf, col0, m0 + q * 32);
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
    if (threadIdx.x == 0) FL_MARK(p, 8);
    cluster_barrier_sync();  // neither CTA's barriers or TMEM go away while the other may use them
    if (threadIdx.x == 0) FL_MARK(p, 9);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

// How many CTA pairs of this kernel can be resident at once.
template <int DT, int BN, int PRO, int KS>
int pair_max_clusters() {
    using C = PairCfg<BN, PRO, KS>;
    auto kern = fl_pair_kernel<DT, BN, PRO, KS, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * KS, 1, 1);
    cfg.blockDim = dim3(PRO != PRO_NONE ? 384 : 256, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * KS;
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

template <int DT, int BN, int PRO, int KS, bool DUAL, bool MULTI>
cudaError_t launch_pair(const ParamsT<MULTI>& p, int grid, cudaStream_t stream) {
    using C = PairCfg<BN, PRO, KS>;
    auto kern = fl_pair_kernel<DT, BN, PRO, KS, DUAL, MULTI>;
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
    attr[0].val.clusterDim.x = 2 * KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = p.pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace fl
