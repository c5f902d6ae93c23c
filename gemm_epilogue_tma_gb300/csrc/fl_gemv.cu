// Decode kernel for one to eight activation rows: the dense layer (and the
// SwiGLU gate/up pair) as a weight-streaming matrix-vector product.
//
// With M <= 8 rows a 128-row tcgen05 MMA is more than 93 % padding and the
// step is bound by reading the weights once from HBM; what decides its time
// is how early the weight stream starts, how many bytes each SM keeps in
// flight, and how little fixed work surrounds it. Here the weights are the
// B operand of warp-level m16n8k16 tensor-core MMAs fed straight from
// registers: each lane loads 16-byte weight vectors (8 consecutive k of one
// row) with non-allocating global loads, in blocks of 8 per lane, double
// buffered so the next block's loads are in flight while the current block's
// MMAs run (the first block is issued before the activation rows arrive).
// The activation rows (at most 8, the A operand's rows 0..7; rows 8..15 are
// zero) come from shared memory. Inside each 32-wide k chunk the MMA's k
// order is a fixed permutation of the physical one, applied identically to
// both operands (lane quad t holds physical k = 8t .. 8t+7 as the MMA's
// k = 2t, 2t+1, 2t+8, 2t+9 of two consecutive MMAs), so a dot product's terms
// are the same; the fp32 accumulation order differs from the tcgen05 kernels'
// but is fixed, so results are bit-reproducible.
//
// The unit of work is a block of 8 weight rows; a CTA's 8 warps split its K
// range into 8 slices and add their partial sums through shared memory in
// warp order. Every CTA builds the prologue-transformed activation rows in
// shared memory (RMSNorm / LayerNorm statistics of the few rows, then the
// fold, rounded once to the dtype as in the tcgen05 kernels). The epilogue
// (RMS row scale, bias, activation, residual; or for the gate/up pair
// h = silu(g) * u) is applied to the reduced sums.
#include "fl_common.cuh"
#include "fl_internal.h"

namespace fl {

namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kVec = 8;      // 16-bit elements per 16-byte vector
constexpr int kChunk = 32;   // k values per MMA pair: 4 lanes x 8
constexpr int kBlock = 8;    // 16-byte weight vectors per lane per register block

// Row stride of the activation rows in shared memory, in elements: a multiple
// of 64 plus 32 (128 k-bytes + 64), so the 8 lanes of a quarter warp (two
// rows, four 16-byte vectors each) hit 32 different banks.
__host__ __device__ __forceinline__ int xs_stride(int K) { return (K + 63) / 64 * 64 + 32; }

// Shared memory of one CTA: the activation rows, then for LayerNorm gamma
// and beta.
__host__ __device__ __forceinline__ int smem_bytes(int M, int K, int pro) {
    return (M * xs_stride(K) + (pro == PRO_LN ? 2 * K : 0)) * 2;
}

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// D[16x8] += A[16x16] B[16x8], fp32 accumulate; A rows 8..15 are zero.
template <int DT>
__device__ __forceinline__ void mma_rows8(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (DT == 0) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    }
}

// One 32-wide k chunk: lane (g, t) holds physical k = 8t .. 8t+7 of its
// activation row (xv) and of its weight row (wv).
template <int DT>
__device__ __forceinline__ void mma_chunk(float (&c)[4], const uint4& xv, const uint4& wv) {
    mma_rows8<DT>(c, xv.x, xv.y, wv.x, wv.y);
    mma_rows8<DT>(c, xv.z, xv.w, wv.z, wv.w);
}

// This warp's slice of the K chunks: [c0, c1).
struct Slice {
    int c0, c1;
};
__device__ __forceinline__ Slice warp_slice(int K, int warp) {
    const int chunks = (K + kChunk - 1) / kChunk, per = (chunks + kGemvWarps - 1) / kGemvWarps;
    const int c0 = min(chunks, warp * per);
    return {c0, min(chunks, c0 + per)};
}

// L2 prefetch of the first register block this lane will read from one
// weight row (before the dependency wait: L2 is the point of coherence, so a
// prefetch cannot bring in stale data even of a tensor the previous kernel
// writes). One block measured best: none 8.98, two blocks 8.37, one 8.19 us
// at M = 1, 4096 x 4096.
__device__ __forceinline__ void prefetch_slice(const uint16_t* row, Slice s, int t) {
    for (int c = s.c0 + 2 * t; c < s.c1 && c < s.c0 + kBlock; c += 8)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + (size_t)c * kChunk));
}

// One block of a warp's weight stream: kBlock / NW consecutive chunks of its
// K slice, for NW weight matrices read with the same activation rows, in
// registers (kBlock 16-byte vectors per lane).
template <int NW>
struct WBlock {
    static constexpr int U = kBlock / NW;
    uint4 w[NW][U];
};

// Issues the loads of block b (chunks s.c0 + b*U ..) of the unit whose
// weight rows (this lane's row g, one per matrix) are rows[]; zeros past K.
template <int NW>
__device__ __forceinline__ void load_block(WBlock<NW>& B, const uint16_t* const (&rows)[NW], int b, Slice s, int K,
                                           int t) {
    constexpr int U = WBlock<NW>::U;
#pragma unroll
    for (int i = 0; i < U; ++i) {
        const int c = s.c0 + b * U + i, k = c * kChunk + 8 * t;
        const bool in = c < s.c1 && k < K;
#pragma unroll
        for (int j = 0; j < NW; ++j) B.w[j][i] = in ? ld_stream(rows[j] + k) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// acc[j] += activation rows . block b of matrix j.
template <int DT, int NW>
__device__ __forceinline__ void mma_block(const WBlock<NW>& B, const uint16_t* xrow, int b, Slice s, int K, int t,
                                          float (&acc)[NW][4]) {
    constexpr int U = WBlock<NW>::U;
#pragma unroll
    for (int i = 0; i < U; ++i) {
        const int c = s.c0 + b * U + i, k = c * kChunk + 8 * t;
        if (c < s.c1) {  // warp-uniform
            const uint4 xv = (xrow != nullptr && k < K) ? *reinterpret_cast<const uint4*>(xrow + k)
                                                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < NW; ++j) mma_chunk<DT>(acc[j], xv, B.w[j][i]);
        }
    }
}

// The units of this CTA (blockIdx.x, + gridDim.x, ..), each an 8-row weight
// block over all of K: this warp streams its K slice of each unit in
// register blocks, the loads of the next block (of this unit or the next)
// issued before the MMAs of the current one, then every warp's partial sums
// go through shared memory (fixed warp order) to finish(unit, lane sums).
// A (block 0 of the first unit) must have been loaded by the caller; mark(s)
// records trace slot s (timing builds only).
// rows_of(u, rows) gives this lane's weight row of each matrix in unit u.
template <int DT, int NW, typename RowsOf, typename Finish, typename Mark>
__device__ __forceinline__ void stream_units(WBlock<NW>& A, int units, int K, const uint16_t* xrow, Slice s,
                                             RowsOf rows_of, float (*red)[kGemvWarps][32][2 * NW], Finish finish,
                                             Mark mark) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3;
    const int nblk = (s.c1 - s.c0 + WBlock<NW>::U - 1) / WBlock<NW>::U;
    WBlock<NW> B;
    int q = 0, buf = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, buf ^= 1) {
        float acc[NW][4] = {};
        for (int b = 0; b < nblk; ++b, ++q) {
            int nu = u, nb = b + 1;
            if (nb == nblk) {
                nu += gridDim.x;
                nb = 0;
            }
            const uint16_t* rows[NW];
            if (nu < units) rows_of(nu, rows);
            if ((q & 1) == 0) {
                if (nu < units) load_block<NW>(B, rows, nb, s, K, t);
                mma_block<DT, NW>(A, xrow, b, s, K, t, acc);
            } else {
                if (nu < units) load_block<NW>(A, rows, nb, s, K, t);
                mma_block<DT, NW>(B, xrow, b, s, K, t, acc);
            }
        }
        // lane (g, t): rows m = g, columns 2t, 2t+1 of each matrix
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            red[buf][warp][lane][2 * j] = acc[j][0];
            red[buf][warp][lane][2 * j + 1] = acc[j][1];
        }
        __syncthreads();
        if (threadIdx.x == 0) mark(u == (int)blockIdx.x ? 3 : 4);
        if (warp == 0) {
            float v[2 * NW];
#pragma unroll
            for (int e = 0; e < 2 * NW; ++e) v[e] = red[buf][0][lane][e];
#pragma unroll
            for (int w = 1; w < kGemvWarps; ++w)
#pragma unroll
                for (int e = 0; e < 2 * NW; ++e) v[e] += red[buf][w][lane][e];
            finish(u, v);
        }
        // (red is double-buffered: the next unit writes the other half, and
        // the one after that only follows the next __syncthreads)
    }
}

// Sum over the CTA of one value per activation row, in a fixed order
// (per-thread partials, warp butterflies, the warps in index order); every
// thread gets the sums in tot[]. Ends with __syncthreads.
template <int R>
__device__ __forceinline__ void row_sums(float (&v)[R], float (*part)[R], float* tot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < R; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[m] += __shfl_xor_sync(0xffffffffu, v[m], o);
        if (lane == 0) part[warp][m] = v[m];
    }
    __syncthreads();
    if (threadIdx.x < R) {
        float a = 0.f;
        for (int w = 0; w < kGemvWarps; ++w) a += part[w][threadIdx.x];
        tot[threadIdx.x] = a;
    }
    __syncthreads();
}

// 16-byte asynchronous copy global -> shared (allocating in L1: the CTAs on
// one SM read the same rows), and the wait
// for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Rows of the prologue-transformed activation, in shared memory: xs[m][k] at
// row stride xs_stride(K), M <= kGemvMaxRows rows; rscale[m] = the RMS row
// scale (else 1). Every thread owns the 16-byte columns c = tid, tid + 256,
// .. of every row. RMSNorm, the input bias and the plain copy load two
// columns of every row (and of gamma / the bias) into registers at a time,
// all before using any, and store the folded values (x * gamma or x + bias,
// rounded once; the RMS scale goes to the epilogue): one memory round trip
// for K <= 4096. LayerNorm needs its rows twice (shifted sums, then the
// fold): up to four rows of K <= 4096 it holds them in registers too; beyond
// that it stages them (and gamma, beta, into the side area after the rows)
// with asynchronous copies, all in flight at once and holding no registers.
// A thread only touches its own columns, so only the row sums need
// barriers. (Asynchronous or bulk-copy staging of the RMSNorm rows measured
// about 1 us slower at K = 4096.)
// R: a bound on M (2, 4 or 8), so the per-row loops unroll to no more rows
// than there can be.
template <int DT, int PRO, int R, typename Pre>
__device__ void build_rows(const GemvParams& p, uint16_t* xs, float* rscale, Pre pre) {
    using Ops = DTypeOps<DT>;
    const int M = p.M, K = p.K, kv = K / kVec, ld = xs_stride(K);
    __shared__ float part[kGemvWarps][R];
    __shared__ float tot[R];
    bool pre_done = false;
    if (PRO != PRO_LN) {
        constexpr int G = 2;
        float sq[R];
#pragma unroll
        for (int m = 0; m < R; ++m) sq[m] = 0.f;
        for (int c0 = threadIdx.x; c0 < kv; c0 += G * kGemvThreads) {
            uint4 v[G][R], gv[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int c = c0 + j * kGemvThreads;
                if (c < kv) {
                    if (PRO != PRO_NONE) gv[j] = ldg_v4(p.gamma + (size_t)c * kVec);
#pragma unroll
                    for (int m = 0; m < R; ++m)
                        if (m < M) v[j][m] = ldg_v4(p.x + (size_t)m * K + (size_t)c * kVec);
                }
            }
            if (!pre_done) {
                pre();
                pre_done = true;
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int c = c0 + j * kGemvThreads;
                if (c < kv) {
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < M) {
                            uint4 o = v[j][m];
                            if (PRO == PRO_RMS) {
                                const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = Ops::unpack(w[e]);
                                    sq[m] = fmaf(f.x, f.x, fmaf(f.y, f.y, sq[m]));
                                }
                                o = make_uint4(Ops::mul2(o.x, gv[j].x), Ops::mul2(o.y, gv[j].y),
                                               Ops::mul2(o.z, gv[j].z), Ops::mul2(o.w, gv[j].w));
                            } else if (PRO == PRO_ADD) {
                                o = make_uint4(Ops::add2(o.x, gv[j].x), Ops::add2(o.y, gv[j].y),
                                               Ops::add2(o.z, gv[j].z), Ops::add2(o.w, gv[j].w));
                            }
                            *reinterpret_cast<uint4*>(xs + (size_t)m * ld + (size_t)c * kVec) = o;
                        }
                    }
                }
            }
        }
        if (!pre_done) pre();
        if (PRO == PRO_RMS) {
            row_sums(sq, part, tot);
            if (threadIdx.x < R) rscale[threadIdx.x] = rsqrtf(tot[threadIdx.x] / (float)K + p.eps);
        } else if (threadIdx.x < R) {
            rscale[threadIdx.x] = 1.f;
        }
        __syncthreads();
        return;
    }
    // LayerNorm: statistics in one pass of shifted sums, d = x - c with c the
    // row's first element (exact for constant rows, no cancellation for rows
    // with a large offset): mean = c + sum(d) / K, var = sum(d^2) / K -
    // (sum(d) / K)^2; every thread derives the rows' mean and 1/sigma from
    // the reduced sums, then folds its own columns.
    const bool has_beta = p.beta != nullptr;
    __shared__ float part2[kGemvWarps][2 * R];
    __shared__ float tot2r[2 * R];
    float cm[R], sv[2 * R];
#pragma unroll
    for (int m = 0; m < R; ++m) {
        cm[m] = m < M ? Ops::unpack((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p.x + (size_t)m * K))).x
                      : 0.f;
        sv[m] = sv[R + m] = 0.f;
    }
    auto stats_of = [&](const uint4& o, int m) {
        const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = Ops::unpack(w[e]);
            const float a = f.x - cm[m], b = f.y - cm[m];
            sv[m] += a + b;
            sv[R + m] = fmaf(a, a, fmaf(b, b, sv[R + m]));
        }
    };
    float mean[R], rstd[R];
    auto finish_stats = [&] {
        row_sums(sv, part2, tot2r);
        const float inv_k = 1.0f / (float)K;
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const float e1 = tot2r[m] * inv_k;
            mean[m] = cm[m] + e1;
            rstd[m] = rsqrtf(fmaxf(tot2r[R + m] * inv_k - e1 * e1, 0.f) + p.eps);
        }
        if (threadIdx.x < R) rscale[threadIdx.x] = 1.f;
    };
    auto fold = [&](uint4 o, const uint4& gv, const uint4& bv, int m) {
        const uint32_t xw[4] = {o.x, o.y, o.z, o.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = Ops::unpack(xw[e]), gg = Ops::unpack(gw[e]), bb = Ops::unpack(bw[e]);
            ow[e] = Ops::pack(fmaf((f.x - mean[m]) * rstd[m], gg.x, bb.x), fmaf((f.y - mean[m]) * rstd[m], gg.y, bb.y));
        }
        return make_uint4(ow[0], ow[1], ow[2], ow[3]);
    };
    if (R <= 4 && kv <= 2 * kGemvThreads) {
        // at most four rows and two columns per thread: rows, gamma and beta in registers,
        // one memory round trip
        uint4 v[2][R], gv[2], bv[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = threadIdx.x + j * kGemvThreads;
            gv[j] = bv[j] = make_uint4(0u, 0u, 0u, 0u);
            if (c < kv) {
                gv[j] = ldg_v4(p.gamma + (size_t)c * kVec);
                if (has_beta) bv[j] = ldg_v4(p.beta + (size_t)c * kVec);
#pragma unroll
                for (int m = 0; m < R; ++m)
                    if (m < M) v[j][m] = ldg_v4(p.x + (size_t)m * K + (size_t)c * kVec);
            }
        }
        pre();
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (threadIdx.x + j * kGemvThreads < kv)
#pragma unroll
                for (int m = 0; m < R; ++m)
                    if (m < M) stats_of(v[j][m], m);
        finish_stats();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = threadIdx.x + j * kGemvThreads;
            if (c < kv)
#pragma unroll
                for (int m = 0; m < R; ++m)
                    if (m < M)
                        *reinterpret_cast<uint4*>(xs + (size_t)m * ld + (size_t)c * kVec) = fold(v[j][m], gv[j], bv[j], m);
        }
        __syncthreads();
        return;
    }
    // more rows or columns: stage them (and gamma, beta into the side area
    // after the rows) with asynchronous copies, all in flight at once
    uint16_t* gs = xs + (size_t)M * ld;
    uint16_t* bs = gs + K;
    for (int c = threadIdx.x; c < kv; c += kGemvThreads) {
        for (int m = 0; m < M; ++m)
            cp_async16(xs + (size_t)m * ld + (size_t)c * kVec, p.x + (size_t)m * K + (size_t)c * kVec);
        cp_async16(gs + (size_t)c * kVec, p.gamma + (size_t)c * kVec);
        if (has_beta) cp_async16(bs + (size_t)c * kVec, p.beta + (size_t)c * kVec);
    }
    pre();
    cp_async_wait_all();
    for (int c = threadIdx.x; c < kv; c += kGemvThreads)
#pragma unroll
        for (int m = 0; m < R; ++m)
            if (m < M) stats_of(*reinterpret_cast<const uint4*>(xs + (size_t)m * ld + (size_t)c * kVec), m);
    finish_stats();
    for (int c = threadIdx.x; c < kv; c += kGemvThreads) {
        const uint4 gv = *reinterpret_cast<const uint4*>(gs + (size_t)c * kVec);
        const uint4 bv =
            has_beta ? *reinterpret_cast<const uint4*>(bs + (size_t)c * kVec) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int m = 0; m < R; ++m) {
            if (m < M) {
                uint4* slot = reinterpret_cast<uint4*>(xs + (size_t)m * ld + (size_t)c * kVec);
                *slot = fold(*slot, gv, bv, m);
            }
        }
    }
    __syncthreads();
}

// DUAL: the SwiGLU gate/up pair, W[0] = Wg and W[1] = Wu, out[0] = h with
// h = silu(g * rs) * (u * rs) (PRO_RMS only).
template <int DT, int PRO, bool DUAL>
__global__ void __launch_bounds__(kGemvThreads, 2) fl_gemv_kernel(const __grid_constant__ GemvParams p) {
    using Ops = DTypeOps<DT>;
    constexpr int NW = DUAL ? 2 : 1;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    __shared__ float rscale[kGemvMaxRows];
    __shared__ float red[2][kGemvWarps][32][2 * NW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int K = p.K, units = p.row0[p.n_out] / 8;
    const Slice s = warp_slice(K, warp);
    // output i, first row n of the 8-row unit u
    auto unit_of = [&](int u, int& oi, int& n) {
        const int r = u * 8;
        oi = 0;
#pragma unroll
        for (int i = 1; i < 4; ++i)
            if (i < p.n_out && r >= p.row0[i]) oi = i;
        n = r - p.row0[oi];
    };
    auto rows_of = [&](int u, const uint16_t* (&rows)[NW]) {
        int oi, n;
        unit_of(u, oi, n);
        rows[0] = p.W[oi] + (size_t)(n + g) * K;
        if constexpr (DUAL) rows[NW - 1] = p.W[1] + (size_t)(n + g) * K;
    };
    if (threadIdx.x == 0) FL_MARK(p, 0);
    const bool first = (int)blockIdx.x < units;
    const uint16_t* rows0[NW] = {};
    // L2 prefetch of the activation rows and gamma / bias first, then of the
    // first weight blocks, so the small reads the prologue waits for are not
    // queued behind the weight stream (prefetches are safe before the
    // dependency wait: L2 is the point of coherence)
    {
        // (each 128-byte line by one CTA of the grid: the others' loads then
        // hit in L2 or on the request already in flight)
        const int xl = (p.M * K * 2 + 127) / 128, gl = PRO != PRO_NONE ? (K * 2 + 127) / 128 : 0;
        for (int i = (int)(threadIdx.x * gridDim.x + blockIdx.x); i < xl + gl; i += kGemvThreads * gridDim.x) {
            const char* a = i < xl ? reinterpret_cast<const char*>(p.x) + (size_t)i * 128
                                   : reinterpret_cast<const char*>(p.gamma) + (size_t)(i - xl) * 128;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
    }
    if (first) {
        rows_of(blockIdx.x, rows0);
#pragma unroll
        for (int j = 0; j < NW; ++j) prefetch_slice(rows0[j], s, t);
    }
    griddep_wait();
    if (threadIdx.x == 0) FL_MARK(p, 1);
    // the activation loads go out first (ahead of the weight stream in the
    // memory queues), then the first weight block, in flight while the rows
    // are built
    WBlock<NW> A;
    auto pre = [&] {
        asm volatile("" ::: "memory");
        if (first) load_block<NW>(A, rows0, 0, s, K, t);
    };
    if (p.M <= 2)
        build_rows<DT, PRO, 2>(p, xs, rscale, pre);
    else if (p.M <= 4)
        build_rows<DT, PRO, 4>(p, xs, rscale, pre);
    else
        build_rows<DT, PRO, kGemvMaxRows>(p, xs, rscale, pre);
    if (threadIdx.x == 0) FL_MARK(p, 2);
    griddep_launch_dependents();
    const uint16_t* xrow = g < p.M ? xs + (size_t)g * xs_stride(K) : nullptr;
    // lane (g, t) finishes output row m = g, columns n0 + 2t, 2t+1
    auto finish = [&](int u, const float (&v)[2 * NW]) {
        if (g >= p.M) return;
        int oi, n0;
        unit_of(u, oi, n0);
        const int m = g, n = n0 + 2 * t, N = p.N[oi];
        const float rs = rscale[m];
        float y0, y1;
        if constexpr (DUAL) {
            y0 = act_apply(ACT_SILU, v[0] * rs) * (v[2] * rs);
            y1 = act_apply(ACT_SILU, v[1] * rs) * (v[3] * rs);
        } else {
            y0 = v[0] * rs;
            y1 = v[1] * rs;
            if (p.bias[oi] != nullptr) {
                const float2 b = Ops::unpack(*reinterpret_cast<const uint32_t*>(p.bias[oi] + n));
                y0 += b.x;
                y1 += b.y;
            }
            y0 = act_apply(p.act[oi], y0);
            y1 = act_apply(p.act[oi], y1);
            if (p.residual != nullptr) {
                const float2 r = Ops::unpack(*reinterpret_cast<const uint32_t*>(p.residual + (size_t)m * N + n));
                y0 += r.x;
                y1 += r.y;
            }
        }
        *reinterpret_cast<uint32_t*>(p.out[oi] + (size_t)m * N + n) = Ops::pack(y0, y1);
    };
    stream_units<DT, NW>(A, units, K, xrow, s, rows_of, red, finish, [&](int slot) { FL_MARK(p, slot); });
    if (threadIdx.x == 0) FL_MARK(p, 5);
}

template <int DT, int PRO, bool DUAL>
cudaError_t gemv_launch(const GemvParams& p, int grid, int smem, int pdl, cudaStream_t stream) {
    auto kern = fl_gemv_kernel<DT, PRO, DUAL>;
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

int gemv_smem_bytes(int M, int K, int pro) { return smem_bytes(M, K, pro); }

cudaError_t launch_gemv(int dt, int pro, bool dual, const GemvParams& p, int sms, int pdl, cudaStream_t stream) {
    const int smem = smem_bytes(p.M, p.K, pro);
    if (p.M < 1 || p.M > kGemvMaxRows || smem > kGemvSmemMax || p.K % 8 != 0) return cudaErrorInvalidValue;
    if (dual && (pro != PRO_RMS || p.n_out != 1)) return cudaErrorInvalidValue;
    for (int i = 0; i < p.n_out; ++i)
        if (p.N[i] % 8 != 0) return cudaErrorInvalidValue;
    // one CTA per 8-row unit, at most as many as are resident at once
    const int units = p.row0[p.n_out] / 8;
    int per_sm = 0;
#define FL_OCC(DT, PRO, DUAL) \
    if (dt == DT && pro == PRO && dual == DUAL) per_sm = resident_ctas(fl_gemv_kernel<DT, PRO, DUAL>, smem);
    FL_OCC(0, 0, false) FL_OCC(0, 1, false) FL_OCC(0, 2, false) FL_OCC(0, 3, false) FL_OCC(0, 1, true)
    FL_OCC(1, 0, false) FL_OCC(1, 1, false) FL_OCC(1, 2, false) FL_OCC(1, 3, false) FL_OCC(1, 1, true)
#undef FL_OCC
    if (per_sm < 1) return cudaErrorInvalidValue;
    int grid = sms * per_sm;
    if (grid > units) grid = units;
#define FL_CASE(DT, PRO, DUAL) \
    if (dt == DT && pro == PRO && dual == DUAL) return gemv_launch<DT, PRO, DUAL>(p, grid, smem, pdl, stream);
    FL_CASE(0, 0, false) FL_CASE(0, 1, false) FL_CASE(0, 2, false) FL_CASE(0, 3, false) FL_CASE(0, 1, true)
    FL_CASE(1, 0, false) FL_CASE(1, 1, false) FL_CASE(1, 2, false) FL_CASE(1, 3, false) FL_CASE(1, 1, true)
#undef FL_CASE
    return cudaErrorInvalidValue;
}

}  // namespace fl
