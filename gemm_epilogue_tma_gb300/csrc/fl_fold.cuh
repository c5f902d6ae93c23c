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

// LayerNorm statistics: merge this thread's chunk of the K block into the
// running moments of its rows. `valid` says whether the chunk lies inside K
// (out-of-range chunks are zero-filled and must not count).
template <int DT>
__device__ __forceinline__ void ln_stats_stage(uint32_t stage, int t, int ni, bool valid, RowMoments (&mo)[8]) {
    using Ops = DTypeOps<DT>;
    if (!valid) return;
    const int j = t & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < ni) {
            const uint4 v = ld_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j));
            const float2 a = Ops::unpack(v.x), b = Ops::unpack(v.y), c = Ops::unpack(v.z), d = Ops::unpack(v.w);
            const float cm = (((a.x + a.y) + (b.x + b.y)) + ((c.x + c.y) + (d.x + d.y))) * 0.125f;
            float q0 = (a.x - cm) * (a.x - cm), q1 = (a.y - cm) * (a.y - cm);
            q0 = fmaf(b.x - cm, b.x - cm, q0);
            q1 = fmaf(b.y - cm, b.y - cm, q1);
            q0 = fmaf(c.x - cm, c.x - cm, q0);
            q1 = fmaf(c.y - cm, c.y - cm, q1);
            q0 = fmaf(d.x - cm, d.x - cm, q0);
            q1 = fmaf(d.y - cm, d.y - cm, q1);
            mo[i] = merge_moments(mo[i], RowMoments{8.f, cm, q0 + q1});
        }
    }
}

// Merge the moments of the 8 lanes that share each row; every lane ends with
// the row's full moments.
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
                // merge in a fixed order (lower lane first) so both partners agree bit for bit
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

// LayerNorm moments of one row's K block (nvalid chunks of 8 lie inside K).
template <int DT>
__device__ __forceinline__ void ln_stats_row(uint32_t stage, int t, int nvalid, RowMoments& mo) {
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
    // out-of-range chunks are zero-filled: they add nothing to the sum
    float part[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        part[j] = ((v[8 * j] + v[8 * j + 1]) + (v[8 * j + 2] + v[8 * j + 3])) +
                  ((v[8 * j + 4] + v[8 * j + 5]) + (v[8 * j + 6] + v[8 * j + 7]));
    const float cnt = 8.f * (float)nvalid;
    const float cm = (((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]))) / cnt;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float q = 0.f;
        if (j < nvalid) {
#pragma unroll
            for (int e = 0; e < 8; ++e) q = fmaf(v[8 * j + e] - cm, v[8 * j + e] - cm, q);
        }
        part[j] = q;
    }
    const float m2 = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
    mo = merge_moments(mo, RowMoments{cnt, cm, m2});
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
