// Norm prologue work on a staged activation tile, shared by the tile and the
// split-K kernels.
//
// The activation stage holds `box_rows` rows of 64 fp16/bf16 (128 bytes, 128B
// swizzle: the 16-byte chunk j of row r sits at chunk position j ^ (r & 7)).
// The 128 transform threads split it by chunks: thread t owns chunk j = t & 7
// of rows t/8 + 16 i, i < box_rows / 16. A warp therefore touches four whole
// rows per access (no bank conflicts), every warp has work even for a 16-row
// decode box, and each thread needs a single 16-byte slice of gamma / beta.
// Per-row RMS sums of squares are merged across the 8 lanes that share a row
// with butterfly shuffles. LayerNorm folds with row statistics computed ahead
// of the GEMM by the statistics kernel.
#pragma once

#include "fl_common.cuh"

namespace fl {

__device__ __forceinline__ uint32_t fold_row_addr(uint32_t stage, int row, int j) {
    return stage + row * 128 + ((j ^ (row & 7)) << 4);
}

// RMS: accumulate x^2 of this thread's chunks into ss[i] and replace the
// chunks by x * gamma (one rounding, as the 16-bit product rounded once).
template <int DT>
__device__ __forceinline__ void fold_rms_stage(uint32_t stage, uint32_t gamma_slice, int t, int ni, float (&ss)[8]) {
    using Ops = DTypeOps<DT>;
    const int j = t & 7;
    const uint4 g = ld_shared_v4(gamma_slice + j * 16);
    uint4 xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ni) xv[i] = ld_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < ni) {
            const float2 a = Ops::unpack(xv[i].x), b = Ops::unpack(xv[i].y), c = Ops::unpack(xv[i].z),
                         d = Ops::unpack(xv[i].w);
            float s0 = a.x * a.x, s1 = a.y * a.y;
            s0 = fmaf(b.x, b.x, s0);
            s1 = fmaf(b.y, b.y, s1);
            s0 = fmaf(c.x, c.x, s0);
            s1 = fmaf(c.y, c.y, s1);
            s0 = fmaf(d.x, d.x, s0);
            s1 = fmaf(d.y, d.y, s1);
            ss[i] += s0 + s1;
            xv[i].x = Ops::mul2(xv[i].x, g.x);
            xv[i].y = Ops::mul2(xv[i].y, g.y);
            xv[i].z = Ops::mul2(xv[i].z, g.z);
            xv[i].w = Ops::mul2(xv[i].w, g.w);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ni) {
            const uint32_t a = fold_row_addr(stage, (t >> 3) + 16 * i, j);
            st_shared_v4(a, xv[i].x, xv[i].y, xv[i].z, xv[i].w);
        }
}

// LayerNorm fold: chunk := (x - mean) * rstd * gamma + beta, in fp32, rounded once.
template <int DT>
__device__ __forceinline__ void fold_ln_stage(uint32_t stage, uint32_t gb_slice, bool has_beta, int t, int ni,
                                              const float (&mean)[8], const float (&rstd)[8]) {
    using Ops = DTypeOps<DT>;
    const int j = t & 7;
    const uint4 gv = ld_shared_v4(gb_slice + j * 16);
    const uint4 bv = has_beta ? ld_shared_v4(gb_slice + 128 + j * 16) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
    float2 g2[4], b2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        g2[q] = Ops::unpack(gw[q]);
        b2[q] = Ops::unpack(bw[q]);
    }
    uint4 xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ni) xv[i] = ld_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < ni) {
            uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // centre first (exact for 16-bit x against an fp32 mean up to one rounding)
                const float2 f = Ops::unpack(xw[q]);
                xw[q] = Ops::pack(fmaf((f.x - mean[i]) * rstd[i], g2[q].x, b2[q].x),
                                  fmaf((f.y - mean[i]) * rstd[i], g2[q].y, b2[q].y));
            }
            st_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j), xw[0], xw[1], xw[2], xw[3]);
        }
    }
}

// ---------------------------------------------------------------------------
// Thread-per-row forms, for folding into tensor memory: thread t of the
// transform warpgroup owns row t (TMEM lane t), reads its 8 chunks (one per
// quarter-warp bank group, no conflicts) and returns the folded row as 32
// packed 32-bit columns in K order, ready for tcgen05.st.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void fold_rms_row(uint32_t stage, uint32_t gamma_slice, int t, float (&ss)[8],
                                             uint32_t (&o)[32]) {
    using Ops = DTypeOps<DT>;
    const int sw = t & 7;
    uint4 xv[8], gv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) xv[j] = ld_shared_v4(stage + t * 128 + ((j ^ sw) << 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) gv[j] = ld_shared_v4(gamma_slice + j * 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 a = Ops::unpack(xv[j].x), b = Ops::unpack(xv[j].y), c = Ops::unpack(xv[j].z),
                     d = Ops::unpack(xv[j].w);
        float s0 = a.x * a.x, s1 = a.y * a.y;
        s0 = fmaf(b.x, b.x, s0);
        s1 = fmaf(b.y, b.y, s1);
        s0 = fmaf(c.x, c.x, s0);
        s1 = fmaf(c.y, c.y, s1);
        s0 = fmaf(d.x, d.x, s0);
        s1 = fmaf(d.y, d.y, s1);
        ss[j] += s0 + s1;
        o[4 * j + 0] = Ops::mul2(xv[j].x, gv[j].x);
        o[4 * j + 1] = Ops::mul2(xv[j].y, gv[j].y);
        o[4 * j + 2] = Ops::mul2(xv[j].z, gv[j].z);
        o[4 * j + 3] = Ops::mul2(xv[j].w, gv[j].w);
    }
}

// LayerNorm, thread-per-row: row t, chunks [J0, J0 + NJ) of the K block :=
// fma(fma(x, rstd, -mean * rstd), gamma, beta) in fp32, one rounding to the
// dtype (the fp32 error stays relative to |mean| * 2^-24, far below it).
// Every shared-memory load (x, gamma, beta) is issued before any result is
// used: under the TMA and MMA traffic of the main loop a load takes a few
// hundred cycles, so the fold costs one such round, not one per chunk.
template <int DT, int NJ, int J0>
__device__ __forceinline__ void fold_ln_row(uint32_t stage, uint32_t gb_slice, bool has_beta, int t, float rstd,
                                            float nmr, uint32_t (&o)[4 * NJ]) {
    using Ops = DTypeOps<DT>;
    const int sw = t & 7;
    uint4 xv[NJ], gv[NJ], bv[NJ];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) xv[jj] = ld_shared_v4(stage + t * 128 + (((J0 + jj) ^ sw) << 4));
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) gv[jj] = ld_shared_v4(gb_slice + (J0 + jj) * 16);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
        bv[jj] = has_beta ? ld_shared_v4(gb_slice + 128 + (J0 + jj) * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        const uint32_t xw[4] = {xv[jj].x, xv[jj].y, xv[jj].z, xv[jj].w};
        const uint32_t gw[4] = {gv[jj].x, gv[jj].y, gv[jj].z, gv[jj].w};
        const uint32_t bw[4] = {bv[jj].x, bv[jj].y, bv[jj].z, bv[jj].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = Ops::unpack(xw[q]), g = Ops::unpack(gw[q]), b = Ops::unpack(bw[q]);
            o[4 * jj + q] =
                Ops::pack(fmaf(fmaf(f.x, rstd, nmr), g.x, b.x), fmaf(fmaf(f.y, rstd, nmr), g.y, b.y));
        }
    }
}

// Sum of the 8 lanes that share a row (RMS).
__device__ __forceinline__ float row_allreduce8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

}  // namespace fl
