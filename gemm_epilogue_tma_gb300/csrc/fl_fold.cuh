// Norm prologue work on a staged activation tile, shared by the tile and the
// split-K kernels.
//
// The activation stage holds `box_rows` rows of 64 fp16/bf16 (128 bytes, 128B
// swizzle: the 16-byte chunk j of row r sits at chunk position j ^ (r & 7)).
// The 128 transform threads split it by chunks: thread t owns chunk j = t & 7
// of rows t/8 + 16 i, i < box_rows / 16. A warp therefore touches four whole
// rows per access (no bank conflicts), every warp has work even for a 16-row
// decode box, and each thread needs a single 16-byte slice of gamma / beta.
// Per-row results (RMS sum of squares, LayerNorm moments) are merged across
// the 8 lanes that share a row with butterfly shuffles.
#pragma once

#include "fl_common.cuh"

namespace fl {

struct RowMoments {  // running count, mean and sum of squared deviations
    float n, mean, m2;
};

// Chan et al.'s pairwise merge of two partial moment sets.
__device__ __forceinline__ RowMoments merge_moments(RowMoments a, RowMoments b) {
    const float n = a.n + b.n;
    if (n == 0.f) return a;
    const float d = b.mean - a.mean;
    const float wb = b.n / n;
    RowMoments r;
    r.n = n;
    r.mean = a.mean + d * wb;
    r.m2 = a.m2 + b.m2 + d * d * a.n * wb;
    return r;
}

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

// LayerNorm statistics, chunk-parallel: this thread's chunk of each of its
// rows is added to per-row shifted sums (see ShiftedSums below); `valid` says
// whether the chunk lies inside K (zero-filled chunks must not count).
struct ShiftedSums;
template <int DT>
__device__ __forceinline__ void ln_sums_stage(uint32_t stage, int t, int ni, bool valid, ShiftedSums (&st)[8]);

// Moments of the 8 lanes that share each row, merged (Chan et al.) in a fixed
// order so every lane ends with the same full-row moments.
__device__ __forceinline__ void ln_stats_allreduce(RowMoments (&mo)[8], int ni) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < ni) {
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                RowMoments other;
                other.n = __shfl_xor_sync(0xffffffffu, mo[i].n, o);
                other.mean = __shfl_xor_sync(0xffffffffu, mo[i].mean, o);
                other.m2 = __shfl_xor_sync(0xffffffffu, mo[i].m2, o);
                mo[i] = (threadIdx.x & o) ? merge_moments(other, mo[i]) : merge_moments(mo[i], other);
            }
        }
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

// LayerNorm moments of one row by shifted sums: with a shift c near the row
// mean (the mean of the row's first 8 elements), accumulate n, S1 = sum(x - c)
// and S2 = sum((x - c)^2) in fp32; then mean = c + S1 / n and
// m2 = S2 - S1^2 / n, whose subtraction loses only about log2(1 + (mean-c)^2 /
// var) bits. One pass per K block, no division per block.
struct ShiftedSums {
    float c, s1, s2, n;
};

template <int DT>
__device__ __forceinline__ void ln_sums_row(uint32_t stage, int t, int nvalid, ShiftedSums& st) {
    using Ops = DTypeOps<DT>;
    if (nvalid <= 0) return;
    const int sw = t & 7;
    float v[64];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 x = ld_shared_v4(stage + t * 128 + ((j ^ sw) << 4));
        const float2 a = Ops::unpack(x.x), b = Ops::unpack(x.y), c = Ops::unpack(x.z), d = Ops::unpack(x.w);
        v[8 * j + 0] = a.x; v[8 * j + 1] = a.y; v[8 * j + 2] = b.x; v[8 * j + 3] = b.y;
        v[8 * j + 4] = c.x; v[8 * j + 5] = c.y; v[8 * j + 6] = d.x; v[8 * j + 7] = d.y;
    }
    if (st.n == 0.f)
        st.c = (((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]))) * 0.125f;
    float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < nvalid) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dlt = v[8 * j + e] - st.c;
                a1[e & 3] += dlt;
                a2[e & 3] = fmaf(dlt, dlt, a2[e & 3]);
            }
        }
    }
    st.s1 += (a1[0] + a1[1]) + (a1[2] + a1[3]);
    st.s2 += (a2[0] + a2[1]) + (a2[2] + a2[3]);
    st.n += 8.f * (float)nvalid;
}

__device__ __forceinline__ RowMoments ln_sums_moments(const ShiftedSums& st) {
    if (st.n == 0.f) return RowMoments{0.f, 0.f, 0.f};
    const float d = st.s1 / st.n;
    return RowMoments{st.n, st.c + d, fmaxf(st.s2 - st.s1 * d, 0.f)};
}

template <int DT>
__device__ __forceinline__ void ln_sums_stage(uint32_t stage, int t, int ni, bool valid, ShiftedSums (&st)[8]) {
    using Ops = DTypeOps<DT>;
    if (!valid) return;
    const int j = t & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < ni) {
            const uint4 x = ld_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j));
            const float2 a = Ops::unpack(x.x), b = Ops::unpack(x.y), c = Ops::unpack(x.z), d = Ops::unpack(x.w);
            if (st[i].n == 0.f) st[i].c = (((a.x + a.y) + (b.x + b.y)) + ((c.x + c.y) + (d.x + d.y))) * 0.125f;
            const float cc = st[i].c;
            const float e0 = a.x - cc, e1 = a.y - cc, e2 = b.x - cc, e3 = b.y - cc;
            const float e4 = c.x - cc, e5 = c.y - cc, e6 = d.x - cc, e7 = d.y - cc;
            st[i].s1 += ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
            st[i].s2 += ((e0 * e0 + e1 * e1) + (e2 * e2 + e3 * e3)) + ((e4 * e4 + e5 * e5) + (e6 * e6 + e7 * e7));
            st[i].n += 8.f;
        }
    }
}

template <int DT>
__device__ __forceinline__ void fold_ln_row(uint32_t stage, uint32_t gb_slice, bool has_beta, int t, float mean,
                                            float rstd, uint32_t (&o)[32]) {
    using Ops = DTypeOps<DT>;
    const int sw = t & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 x = ld_shared_v4(stage + t * 128 + ((j ^ sw) << 4));
        const uint4 g = ld_shared_v4(gb_slice + j * 16);
        const uint4 b = has_beta ? ld_shared_v4(gb_slice + 128 + j * 16) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, gw[4] = {g.x, g.y, g.z, g.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = Ops::unpack(xw[q]), g2 = Ops::unpack(gw[q]), b2 = Ops::unpack(bw[q]);
            o[4 * j + q] = Ops::pack(fmaf((f.x - mean) * rstd, g2.x, b2.x), fmaf((f.y - mean) * rstd, g2.y, b2.y));
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
