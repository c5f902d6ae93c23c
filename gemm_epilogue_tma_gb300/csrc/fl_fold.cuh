// Prologue work on a staged activation tile (RMSNorm, LayerNorm, input bias),
// shared by the tile, CTA-pair and split-K kernels.
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

// s0 += lo^2, s1 += hi^2 for the two 16-bit values of u, without widening
// them first: the mixed-precision FMA (fp32 result and addend, 16-bit
// factors; sm_100 and later) squares exactly in fp32 and rounds once, the same
// value as fmaf on the widened inputs, in one instruction per element.
template <int DT>
__device__ __forceinline__ void sq_acc2(uint32_t u, float& s0, float& s1) {
    if (DT == DT_F16)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "fma.rn.f32.f16 %0, lo, lo, %0;\n\tfma.rn.f32.f16 %1, hi, hi, %1;\n\t}"
            : "+f"(s0), "+f"(s1)
            : "r"(u));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "fma.rn.f32.bf16 %0, lo, lo, %0;\n\tfma.rn.f32.bf16 %1, hi, hi, %1;\n\t}"
            : "+f"(s0), "+f"(s1)
            : "r"(u));
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
            float s0 = 0.f, s1 = 0.f;
            sq_acc2<DT>(xv[i].x, s0, s1);
            sq_acc2<DT>(xv[i].y, s0, s1);
            sq_acc2<DT>(xv[i].z, s0, s1);
            sq_acc2<DT>(xv[i].w, s0, s1);
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

// Input-bias fold: chunk := x + b (b along K), rounded once to the dtype.
template <int DT>
__device__ __forceinline__ void fold_add_stage(uint32_t stage, uint32_t b_slice, int t, int ni) {
    using Ops = DTypeOps<DT>;
    const int j = t & 7;
    const uint4 b = ld_shared_v4(b_slice + j * 16);
    uint4 xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ni) xv[i] = ld_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ni)
            st_shared_v4(fold_row_addr(stage, (t >> 3) + 16 * i, j), Ops::add2(xv[i].x, b.x), Ops::add2(xv[i].y, b.y),
                         Ops::add2(xv[i].z, b.z), Ops::add2(xv[i].w, b.w));
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
// transform warpgroup owns row t (TMEM lane t), reads chunks [j0, j0 + NJ) of
// its row (one per quarter-warp bank group, no conflicts) and returns them
// folded as 4 * NJ packed 32-bit columns in K order, ready for tcgen05.st.
//
// Each fold is split into a load part, which issues every shared-memory load
// the fold needs (x, gamma and, for LayerNorm, beta), and a compute part, so a
// caller can keep the loads of the next K block in flight while it computes
// and stores this one: under the TMA and MMA traffic of the main loop a shared
// load takes a few hundred cycles.
// ---------------------------------------------------------------------------
template <int NJ, bool LN>
struct FoldRegs {
    uint4 x[NJ];
    uint4 g[NJ];
    uint4 b[LN ? NJ : 1];
};

template <int NJ, bool LN>
__device__ __forceinline__ void fold_row_load(FoldRegs<NJ, LN>& r, uint32_t stage, uint32_t gb_slice, bool has_beta,
                                              int t, int j0) {
    const int sw = t & 7;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) r.x[jj] = ld_shared_v4(stage + t * 128 + (((j0 + jj) ^ sw) << 4));
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) r.g[jj] = ld_shared_v4(gb_slice + (j0 + jj) * 16);
    if (LN) {
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj)
            r.b[jj] = has_beta ? ld_shared_v4(gb_slice + 128 + (j0 + jj) * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// RMS: ss[jj] += sum of x^2 over chunk jj; the chunk := x * gamma (one
// rounding, as the 16-bit product rounded once).
template <int DT, int NJ>
__device__ __forceinline__ void fold_rms_compute(const FoldRegs<NJ, false>& r, float (&ss)[NJ],
                                                 uint32_t (&o)[4 * NJ]) {
    using Ops = DTypeOps<DT>;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        float s0 = 0.f, s1 = 0.f;
        sq_acc2<DT>(r.x[j].x, s0, s1);
        sq_acc2<DT>(r.x[j].y, s0, s1);
        sq_acc2<DT>(r.x[j].z, s0, s1);
        sq_acc2<DT>(r.x[j].w, s0, s1);
        ss[j] += s0 + s1;
        o[4 * j + 0] = Ops::mul2(r.x[j].x, r.g[j].x);
        o[4 * j + 1] = Ops::mul2(r.x[j].y, r.g[j].y);
        o[4 * j + 2] = Ops::mul2(r.x[j].z, r.g[j].z);
        o[4 * j + 3] = Ops::mul2(r.x[j].w, r.g[j].w);
    }
}

// Input bias: chunk := x + b (the bias slice sits where gamma would).
template <int DT, int NJ>
__device__ __forceinline__ void fold_add_compute(const FoldRegs<NJ, false>& r, uint32_t (&o)[4 * NJ]) {
    using Ops = DTypeOps<DT>;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        o[4 * j + 0] = Ops::add2(r.x[j].x, r.g[j].x);
        o[4 * j + 1] = Ops::add2(r.x[j].y, r.g[j].y);
        o[4 * j + 2] = Ops::add2(r.x[j].z, r.g[j].z);
        o[4 * j + 3] = Ops::add2(r.x[j].w, r.g[j].w);
    }
}

// LayerNorm: chunk := fma(fma(x, rstd, -mean * rstd), gamma, beta) in fp32,
// one rounding to the dtype (the fp32 error stays relative to
// |mean| * 2^-24, far below it). Element pairs go through the paired fp32
// FMA: the fold's arithmetic sits on the main loop's critical path.
template <int DT, int NJ>
__device__ __forceinline__ void fold_ln_compute(const FoldRegs<NJ, true>& r, float rstd, float nmr,
                                                uint32_t (&o)[4 * NJ]) {
    using Ops = DTypeOps<DT>;
    const float2 r2 = make_float2(rstd, rstd), n2 = make_float2(nmr, nmr);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        const uint32_t xw[4] = {r.x[jj].x, r.x[jj].y, r.x[jj].z, r.x[jj].w};
        const uint32_t gw[4] = {r.g[jj].x, r.g[jj].y, r.g[jj].z, r.g[jj].w};
        const uint32_t bw[4] = {r.b[jj].x, r.b[jj].y, r.b[jj].z, r.b[jj].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = Ops::unpack(xw[q]), g = Ops::unpack(gw[q]), b = Ops::unpack(bw[q]);
            const float2 y = ffma2(ffma2(f, r2, n2), g, b);
            o[4 * jj + q] = Ops::pack(y.x, y.y);
        }
    }
}

// Whole-row RMS fold (chunks 0-7), loads issued before any use.
template <int DT>
__device__ __forceinline__ void fold_rms_row(uint32_t stage, uint32_t gamma_slice, int t, float (&ss)[8],
                                             uint32_t (&o)[32]) {
    FoldRegs<8, false> r;
    fold_row_load(r, stage, gamma_slice, false, t, 0);
    fold_rms_compute<DT>(r, ss, o);
}

// Whole-row input-bias fold (chunks 0-7), loads issued before any use.
template <int DT>
__device__ __forceinline__ void fold_add_row(uint32_t stage, uint32_t b_slice, int t, uint32_t (&o)[32]) {
    FoldRegs<8, false> r;
    fold_row_load(r, stage, b_slice, false, t, 0);
    fold_add_compute<DT>(r, o);
}

// LayerNorm fold of chunks [J0, J0 + NJ) of row t, loads issued before any use.
template <int DT, int NJ, int J0>
__device__ __forceinline__ void fold_ln_row(uint32_t stage, uint32_t gb_slice, bool has_beta, int t, float rstd,
                                            float nmr, uint32_t (&o)[4 * NJ]) {
    FoldRegs<NJ, true> r;
    fold_row_load(r, stage, gb_slice, has_beta, t, J0);
    fold_ln_compute<DT>(r, rstd, nmr, o);
}

// Sum of the 8 lanes that share a row (RMS).
__device__ __forceinline__ float row_allreduce8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

}  // namespace fl
