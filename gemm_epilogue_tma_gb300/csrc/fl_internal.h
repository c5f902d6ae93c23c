// Declarations shared by the C-ABI host layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fl {

// Prologues applied to the staged activation: none, RMSNorm, LayerNorm, or
// the elementwise input bias (x + b, b along K).
enum Prologue : int { PRO_NONE = 0, PRO_RMS = 1, PRO_LN = 2, PRO_ADD = 3 };
enum ActKind : int { ACT_NONE = 0, ACT_GELU = 1, ACT_SILU = 2, ACT_RELU = 3 };
enum DTypeTag : int { DT_F16 = 0, DT_BF16 = 1 };

// Device status word values (low byte = code; the next byte says which wait gave up).
constexpr int kStatusTimeout = 6;
// Status words per device: one per stream handle in first-use order; word 0
// also serves the legacy default stream and every stream past the table.
constexpr int kStatusSlots = 64;

// CTA tile: 128 rows of the activation; 64 fp16/bf16 along K per stage (one
// 128-byte swizzle row).
constexpr int kBM = 128;
constexpr int kBK = 64;

// Outputs one launch may write: several weights applied to the same
// (normalised) activation, side by side along N (horizontal fusion).
#ifndef FL_MAX_OUT_PARAMS
#define FL_MAX_OUT_PARAMS 4
#endif
constexpr int kMaxOut = FL_MAX_OUT_PARAMS;

// Parameters of one launch. Passed by value as a __grid_constant__ so the
// tensor maps sit in parameter space, where TMA may read them. The first
// output's fields are here; a launch with several outputs passes
// GemmParamsMulti, which appends the others (a single-output launch keeps the
// smaller block: parameter bytes cost launch time on short kernels, 1.5 us on
// the 512 x 1024 x 1024 GEMM).
struct GemmParams {
    CUtensorMap tmA;      // activation [M, K], box {64, 128}, 128B swizzle
    CUtensorMap tmB;      // weight of output 0 [N, K], box {64, BN}, 128B swizzle
    CUtensorMap tmB2;     // second weight [N, K] of the gate/up kernel (else unused)
    CUtensorMap tmOut;    // output 0 [M, N], box {64, 32}, 128B swizzle
    CUtensorMap tmGamma;  // gamma (RMS, LayerNorm) or the input bias, as a [1, K] matrix, box {64, 1}
    CUtensorMap tmBeta;   // beta as a [1, K] matrix, box {64, 1} (LayerNorm with beta)
    const void* bias;      // output 0 bias [N] or null
    const void* residual;  // [M, N] or null (single-output launches only)
    const void* gamma;     // [K] (prologues)
    const void* beta;      // [K] or null (LayerNorm)
    const void* a_ptr;     // activation [M, K]
    const void* ln_stats;  // LayerNorm: float2 (mean, 1/sqrt(var + eps)) per activation row
    void* out_ptr;         // output 0 [M, N] (split-K kernel stores directly)
    int* status;           // the launching stream's device status word
    unsigned long long timeout_ns;
    int M, N, K;           // N: columns of output 0
    int act;               // activation of output 0
    int n_out;             // outputs of this launch (1 .. kMaxOut)
    // first column block (in tiles of this launch's width) of each output;
    // nb0[n_out] is the total, num_n_blocks
    int nb0[kMaxOut + 1];
    int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
    float eps;
    int splits;    // split-K kernel: CTAs per cluster, one K range each
    int kps;       // split-K kernel: 64-wide K blocks per split
    int a_rows;    // split-K kernel: rows of the activation box (128, or M rounded up to 16)
    int pdl;       // launch with a programmatic dependency on the previous kernel of the stream
    // split-K reduction exchange, laid out on the host (tile columns in
    // 8-column chunks, rank r owning chunks [xc_c0[r], xc_c0[r + 1]))
    int w_preload;               // weights may be read before the programmatic dependency resolves
    int s_one_per_sm;           // split-K kernel: the ring leaves room for one CTA per SM only
    int s_stages;                // split-K kernel: pipeline stages of the ring
    int s_stage_bytes;           // split-K kernel: bytes per stage (activation box + weight tile)
    int xc_stride;              // floats per exchange slot row
    unsigned char xc_owner[32];  // owning rank of each chunk
    unsigned char xc_pos[32];    // chunk's position within its owner's slice
    unsigned char xc_c0[12];     // first chunk of each rank; [splits] = chunk count
    float inv_k;                 // 1 / K
    unsigned long long* trace;  // phase timestamps, builds with FL_TRACE only (else unused, null)
};

// Outputs 1 .. n_out - 1 of a multi-output launch.
struct GemmParamsMulti : GemmParams {
    CUtensorMap tmBx[kMaxOut - 1];
    CUtensorMap tmOutx[kMaxOut - 1];
    const void* biasx[kMaxOut - 1];
    void* out_ptrx[kMaxOut - 1];
    int Nx[kMaxOut - 1];
    int actx[kMaxOut - 1];
};

template <bool MULTI>
struct ParamsOf {
    using type = GemmParams;
};
template <>
struct ParamsOf<true> {
    using type = GemmParamsMulti;
};
template <bool MULTI>
using ParamsT = typename ParamsOf<MULTI>::type;

// Records a status message for fl_last_error() on this thread; returns status.
int set_last_error(int status, const char* message);

// LayerNorm row statistics of x [M, K] into stats (M float2: mean, rstd).
cudaError_t launch_ln_stats(int dt, const void* x, int M, int K, float eps, void* stats, int pdl, int sms,
                            cudaStream_t stream);

// Decode kernel (M <= kGemvMaxRows activation rows; the transformed rows
// must fit in kGemvSmemMax bytes of shared memory: gemv_smem_bytes).
constexpr int kGemvMaxRows = 8;
constexpr int kGemvSmemMax = 96 * 1024;

struct GemvParams {
    const uint16_t* x;          // [M, K]
    const uint16_t* gamma;      // RMS / LayerNorm gamma, or the input bias (PRO_ADD)
    const uint16_t* beta;       // LayerNorm beta or null
    const uint16_t* W[4];       // output i: weight [N_i, K] (gate/up pair: W[0] = Wg, W[1] = Wu)
    const uint16_t* bias[4];    // output i: bias [N_i] or null
    uint16_t* out[4];           // output i: [M, N_i]
    int N[4], act[4];
    int row0[5];                // first weight row of each output in the combined row space; row0[n_out] = total
    int n_out;
    const uint16_t* residual;   // [M, N_0] or null (single output)
    int M, K;
    float eps;
    unsigned long long* trace;  // phase timestamps, builds with FL_TRACE only (else unused, null)
};

int gemv_smem_bytes(int M, int K, int pro);
// dual: the SwiGLU gate/up pair (pro = PRO_RMS, one output h = silu(g) * u).
cudaError_t launch_gemv(int dt, int pro, bool dual, const GemvParams& p, int sms, int pdl, cudaStream_t stream);

// Standalone RMSNorm y = x * gamma / sqrt(mean(x^2) + eps) of x [M, K].
cudaError_t launch_rms_norm(int dt, const void* x, const void* gamma, void* y, int M, int K, float eps, int pdl,
                            int sms, cudaStream_t stream);

// Kernel launchers, explicitly instantiated in the kernel translation units.
template <int DT, int BN, int PRO, bool DUAL, bool MULTI = false>
cudaError_t launch_gemm(const ParamsT<MULTI>& p, int grid, cudaStream_t stream);

template <int DT, int BN, int PRO, bool DUAL = false, bool MULTI = false>
cudaError_t launch_splitk(const ParamsT<MULTI>& p, int grid, int splits, cudaStream_t stream);

template <int DT, int BN, int PRO, bool DUAL = false>
int splitk_max_clusters(int splits, int smem_bytes);

template <int DT, int BN, int PRO, int KS, bool DUAL, bool MULTI = false>
cudaError_t launch_pair(const ParamsT<MULTI>& p, int grid, cudaStream_t stream);

template <int DT, int BN, int PRO, int KS>
int pair_max_clusters();

// Shared-memory layout of the split-K kernel: a fixed block of barriers and
// small buffers, then the ring, sized at launch from the activation box
// height (a decode step stages 16 activation rows, not 128), so small-M
// instances fit two CTAs per SM and the next kernel's CTAs can be resident
// (prefetching their weights) while this one finishes.
//
// DUAL (SwiGLU gate/up): every stage holds a tile of Wg and one of Wu after the
// activation box, the MMA fills two accumulators (gate in TMEM columns
// [0, BN), up in [BN, 2 BN)), and the exchange carries both per chunk.
template <int BN, bool DUAL = false>
struct SplitCfg {
    static constexpr int A_MAX_BYTES = kBM * kBK * 2;  // what one MMA reads of A (128 rows)
    static constexpr int NW = DUAL ? 2 : 1;            // weight tiles per stage
    static constexpr int B_BYTES = BN * kBK * 2;       // one weight tile
    static constexpr int STAGE_B_BYTES = NW * B_BYTES;
    static constexpr int MAX_STAGES = 8;
    static constexpr int TMEM_COLS = NW * BN < 32 ? 32 : NW * BN;
    static constexpr int CHUNK_FLOATS = 8 * NW;        // floats of one 8-column chunk in an exchange slot
    static constexpr int NUM_BARS = 3 * MAX_STAGES + 4;
    static constexpr int OFF_BAR = 0;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_SS = (OFF_SLOT + 16 + 15) / 16 * 16;   // [128] partial sum of squares
    static constexpr int OFF_GB = (OFF_SS + kBM * 4 + 127) / 128 * 128;
    static constexpr int OFF_RING = (OFF_GB + MAX_STAGES * 256 + 1023) / 1024 * 1024;
    // Ring budgets: two CTAs per SM, else one.
    static constexpr int RING_SMALL = 100 * 1024;
    static constexpr int RING_LARGE = 192 * 1024;
    // Reduction exchange (in the ring once the main loop is over). Rank r of
    // the cluster owns the 8-column chunks [r C / s, (r + 1) C / s) of the
    // tile (C = BN / 8 chunks, s ranks). A slot holds one rank's fp32 partial
    // of one owner's columns, `rows` rows of xchg_stride(s) floats: the widest
    // slice plus 4 (the first of them carries the row's partial sum of
    // squares). An owner receives s slots (its own included), a sender keeps
    // s - 1 outgoing ones. A stride of 4 mod 8 words keeps rows on distinct
    // banks for 16-byte accesses.
    static constexpr int CHUNKS = BN / 8;
    __host__ __device__ static constexpr int xchg_stride(int s) { return (CHUNKS + s - 1) / s * CHUNK_FLOATS + 4; }
    __host__ __device__ static constexpr int xchg_bytes(int s, int rows) {
        return (2 * s - 1) * rows * xchg_stride(s) * 4;
    }
    static constexpr bool xchg_fits_large() {
        for (int s = 1; s <= 8; ++s)
            if (xchg_bytes(s, kBM) > RING_LARGE / (kBM * 128 + STAGE_B_BYTES) * (kBM * 128 + STAGE_B_BYTES))
                return false;
        return true;
    }
    // (single weight: every cluster size fits; the gate/up form's exchange is
    // twice as wide, and the host lowers its split until it fits)
    static_assert(DUAL || xchg_fits_large(), "the reduction exchange must fit in the large ring");
    // dynamic shared memory of a launch: fixed block, ring, room for one
    // MMA's 128-row read of A from the last stage, alignment slack
    __host__ __device__ static constexpr int smem_bytes(int stages, int stage_bytes) {
        return OFF_RING + stages * stage_bytes + (stage_bytes < A_MAX_BYTES ? A_MAX_BYTES - stage_bytes : 0) + 1024;
    }
    static constexpr int SMEM_MAX = OFF_RING + RING_LARGE + 1024 + 16 * 1024;
};

// Ring geometry of one split-K launch (host side).
struct SplitGeom {
    int stages, stage_bytes, smem_bytes;
};

// Shared-memory bytes of each tile configuration (host-visible).
template <int BN, bool DUAL>
struct TileCfg {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES * (DUAL ? 2 : 1);
    static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int ACC_COLS = BN * (DUAL ? 2 : 1);  // one accumulator buffer
    static constexpr int TMEM_COLS = 2 * ACC_COLS;         // double buffered
    static constexpr int EPI_WARPS = 4;
    static constexpr int EPI_BUF_BYTES = 32 * 128;         // 32 rows x 64 cols x 2 B per warp
    static constexpr int OFF_EPI = STAGES * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUF_BYTES;
    static constexpr int NUM_BARS = 3 * STAGES + 6 + 1;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ROWSCALE = (OFF_SLOT + 16 + 15) / 16 * 16;
    // per stage: the gamma and beta slices of the K block (64 x 2 B each)
    static constexpr int OFF_GB = (OFF_ROWSCALE + 2 * kBM * 4 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = OFF_GB + STAGES * 256 + 1024;  // + alignment slack
};

}  // namespace fl
