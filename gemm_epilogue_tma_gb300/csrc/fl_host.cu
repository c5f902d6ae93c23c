// C-ABI host layer of libfusedlin: argument validation, TMA tensor-map
// encoding, variant dispatch, and the device status word.
//
// Validation is pure host code and runs before any CUDA call, so a rejected
// call neither launches nor writes anything (and can be tested without a GPU).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cstdlib>
#include <mutex>

#include "../../include/fusedlin.h"
#include "fl_internal.h"

using fl::GemmParams;
using fl::GemmParamsMulti;

// Device status words: a kernel records a bounded-wait expiry in the word of
// the stream it was launched (or captured) on.
__device__ int g_fl_status[fl::kStatusSlots];

namespace {

thread_local char tls_err[512] = "";

fl_status fail(fl_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(tls_err, sizeof(tls_err), fmt, ap);
    va_end(ap);
    return s;
}

fl_status ok() {
    tls_err[0] = '\0';
    return FL_OK;
}

std::atomic<int> g_opt_tile_n{0};
std::atomic<int> g_opt_variant{0};
std::atomic<int> g_opt_timeout_ms{2000};
std::atomic<int> g_opt_split_k{0};
std::atomic<int> g_opt_pdl{1};
std::atomic<int> g_opt_preload{0};
std::atomic<int> g_opt_cache{1};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// ---------------------------------------------------------------------------
// device information (cached per device)
// ---------------------------------------------------------------------------
struct DeviceInfo {
    // set (release) once every field below is filled; read (acquire) before
    // any of them, so a thread that sees it set also sees the fields
    std::atomic<bool> ready{false};
    int sms = 0;
    int major = 0, minor = 0;
    int* status = nullptr;  // device address of g_fl_status[0]
    // stream handle of each status word (word 0: the legacy default stream
    // and overflow), filled in first-use order under slot_mu
    std::mutex slot_mu;
    cudaStream_t slot_stream[fl::kStatusSlots] = {};
    int slots_used = 1;
    // stream-ordered pool for per-call scratch (LayerNorm row statistics);
    // the library's own, so the process's default pool keeps its settings
    cudaMemPool_t pool = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

fl_status device_info(DeviceInfo** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(FL_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(FL_ERR_UNSUPPORTED, "device index %d out of range", dev);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            cudaDeviceProp prop;
            e = cudaGetDeviceProperties(&prop, dev);
            if (e != cudaSuccess) return fail(FL_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
            d.sms = prop.multiProcessorCount;
            d.major = prop.major;
            d.minor = prop.minor;
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_fl_status);
            if (e != cudaSuccess) return fail(FL_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            e = cudaMemPoolCreate(&d.pool, &props);
            if (e != cudaSuccess) return fail(FL_ERR_CUDA, "cudaMemPoolCreate: %s", cudaGetErrorString(e));
            // keep freed scratch in the pool instead of returning it at every synchronisation
            uint64_t keep = 64ull << 20;
            cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            d.ready.store(true, std::memory_order_release);
        }
    }
    if (!(d.major == 10 && d.minor == 3))
        return fail(FL_ERR_UNSUPPORTED, "needs a compute capability 10.3 (sm_103a) device, found %d.%d", d.major,
                    d.minor);
    *out = &d;
    return FL_OK;
}

int device_index() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

// Index of the status word of `stream` (see DeviceInfo::slot_stream). A thread
// keeps its last answer, so a loop on one stream takes the lock once.
int status_slot(DeviceInfo* di, cudaStream_t stream) {
    thread_local const DeviceInfo* last_di = nullptr;
    thread_local cudaStream_t last_stream = nullptr;
    thread_local int last_slot = 0;
    if (stream == nullptr) return 0;
    if (last_di == di && last_stream == stream) return last_slot;
    int i = 1;
    {
        std::lock_guard<std::mutex> lk(di->slot_mu);
        while (i < di->slots_used && di->slot_stream[i] != stream) ++i;
        if (i == di->slots_used && i < fl::kStatusSlots) {
            di->slot_stream[i] = stream;
            di->slots_used = i + 1;
        }
    }
    if (i >= fl::kStatusSlots) i = 0;
    last_di = di;
    last_stream = stream;
    last_slot = i;
    return i;
}

int* stream_status(DeviceInfo* di, cudaStream_t stream) { return di->status + status_slot(di, stream); }

// ---------------------------------------------------------------------------
// TMA tensor maps
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Row-major [outer, inner] fp16/bf16 matrix, box {box_inner, box_outer},
// 128-byte swizzle (or none), zero fill out of range.
fl_status encode_2d(CUtensorMap* m, int dt, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer, bool swizzle = true) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return fail(FL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt == FL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%llu, %llu] matrix, box {%u, %u}", (int)r,
                    (unsigned long long)outer, (unsigned long long)inner, box_inner, box_outer);
    return FL_OK;
}

// ---------------------------------------------------------------------------
// outputs of one launch
// ---------------------------------------------------------------------------
// One or more outputs computed from the same (prologue-transformed)
// activation: output i = act_i(A' W_i^T + bias_i), laid side by side along N.
struct OutDesc {
    const void* W;     // [N, K]
    const void* bias;  // [N] or null
    void* out;         // [M, N]
    int N;
    int act;
};
struct Outs {
    int n = 0;
    OutDesc o[fl::kMaxOut];
};

Outs single_out(const void* W, const void* bias, void* out, int N, int act) {
    Outs r;
    r.n = 1;
    r.o[0] = OutDesc{W, bias, out, N, act};
    return r;
}

// Column blocks of width b over all outputs (each output starts a new block).
long long nblocks(const Outs& outs, int b) {
    long long n = 0;
    for (int i = 0; i < outs.n; ++i) n += (outs.o[i].N + b - 1) / b;
    return n;
}

// Per-output parameters of a launch whose tiles are `width` columns wide.
// The weight maps have boxes of `b_rows` rows. Output 0 goes to the base
// block, the others to the multi-output extension.
fl_status fill_outputs(GemmParamsMulti& p, int dt, const Outs& outs, int M, int K, int width, int b_rows) {
    fl_status st;
    p.n_out = outs.n;
    int nb = 0;
    for (int i = 0; i < outs.n; ++i) {
        const OutDesc& o = outs.o[i];
        CUtensorMap* tb = i == 0 ? &p.tmB : &p.tmBx[i - 1];
        CUtensorMap* to = i == 0 ? &p.tmOut : &p.tmOutx[i - 1];
        if ((st = encode_2d(tb, dt, o.W, K, o.N, fl::kBK, b_rows)) != FL_OK) return st;
        if ((st = encode_2d(to, dt, o.out, o.N, M, 64, 32)) != FL_OK) return st;
        (i == 0 ? p.bias : p.biasx[i - 1]) = o.bias;
        (i == 0 ? p.out_ptr : p.out_ptrx[i - 1]) = o.out;
        (i == 0 ? p.N : p.Nx[i - 1]) = o.N;
        (i == 0 ? p.act : p.actx[i - 1]) = o.act;
        p.nb0[i] = nb;
        nb += (o.N + width - 1) / width;
    }
    for (int i = outs.n; i <= fl::kMaxOut; ++i) p.nb0[i] = nb;
    p.num_n_blocks = nb;
    return FL_OK;
}

// ---------------------------------------------------------------------------
// tile kernel dispatch
// ---------------------------------------------------------------------------
cudaError_t dispatch_tile(int dt, int bn, int pro, bool dual, const GemmParamsMulti& p, int grid, cudaStream_t s) {
    const bool multi = p.n_out > 1;
#define FL_CASE(DT, BN, PRO, DUAL) \
    if (dt == DT && bn == BN && pro == PRO && dual == DUAL && !multi) return fl::launch_gemm<DT, BN, PRO, DUAL>(p, grid, s);
    FL_CASE(0, 128, 0, false) FL_CASE(0, 256, 0, false) FL_CASE(0, 128, 1, false) FL_CASE(0, 256, 1, false)
    FL_CASE(0, 128, 2, false) FL_CASE(0, 256, 2, false) FL_CASE(0, 128, 3, false) FL_CASE(0, 256, 3, false)
    FL_CASE(0, 128, 1, true)
    FL_CASE(1, 128, 0, false) FL_CASE(1, 256, 0, false) FL_CASE(1, 128, 1, false) FL_CASE(1, 256, 1, false)
    FL_CASE(1, 128, 2, false) FL_CASE(1, 256, 2, false) FL_CASE(1, 128, 3, false) FL_CASE(1, 256, 3, false)
    FL_CASE(1, 128, 1, true)
#undef FL_CASE
#define FL_CASE(DT, BN, PRO) \
    if (dt == DT && bn == BN && pro == PRO && !dual && multi) return fl::launch_gemm<DT, BN, PRO, false, true>(p, grid, s);
    FL_CASE(0, 128, 1) FL_CASE(0, 256, 1) FL_CASE(0, 128, 2) FL_CASE(0, 256, 2)
    FL_CASE(1, 128, 1) FL_CASE(1, 256, 1) FL_CASE(1, 128, 2) FL_CASE(1, 256, 2)
#undef FL_CASE
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_splitk(int dt, int bn, int pro, bool dual, const GemmParamsMulti& p, int grid, int splits,
                            cudaStream_t s) {
    if (p.n_out > 1) {
#define FL_CASE(DT, BN, PRO) \
        if (dt == DT && bn == BN && pro == PRO && !dual)   \
            return fl::launch_splitk<DT, BN, PRO, false, true>(p, grid, splits, s);
        FL_CASE(0, 64, 1) FL_CASE(0, 64, 2) FL_CASE(0, 128, 1) FL_CASE(0, 128, 2)
        FL_CASE(1, 64, 1) FL_CASE(1, 64, 2) FL_CASE(1, 128, 1) FL_CASE(1, 128, 2)
#undef FL_CASE
        return cudaErrorInvalidValue;
    }
    if (dual) {
        if (pro != fl::PRO_RMS) return cudaErrorInvalidValue;
        if (bn == 64) return dt == 0 ? fl::launch_splitk<0, 64, fl::PRO_RMS, true>(p, grid, splits, s)
                                     : fl::launch_splitk<1, 64, fl::PRO_RMS, true>(p, grid, splits, s);
        if (bn == 128) return dt == 0 ? fl::launch_splitk<0, 128, fl::PRO_RMS, true>(p, grid, splits, s)
                                      : fl::launch_splitk<1, 128, fl::PRO_RMS, true>(p, grid, splits, s);
        return cudaErrorInvalidValue;
    }
#define FL_CASE(DT, BN, PRO) \
    if (dt == DT && bn == BN && pro == PRO) return fl::launch_splitk<DT, BN, PRO>(p, grid, splits, s);
    FL_CASE(0, 64, 0) FL_CASE(0, 64, 1) FL_CASE(0, 64, 2) FL_CASE(0, 64, 3)
    FL_CASE(0, 128, 0) FL_CASE(0, 128, 1) FL_CASE(0, 128, 2) FL_CASE(0, 128, 3)
    FL_CASE(1, 64, 0) FL_CASE(1, 64, 1) FL_CASE(1, 64, 2) FL_CASE(1, 64, 3)
    FL_CASE(1, 128, 0) FL_CASE(1, 128, 1) FL_CASE(1, 128, 2) FL_CASE(1, 128, 3)
#undef FL_CASE
    return cudaErrorInvalidValue;
}

// Largest row count whose SwiGLU gate/up GEMM takes the split-K form.
constexpr int kDualSplitRows = 64;

// Split-K plan for shapes with too few output tiles to fill the GPU: 64-wide
// weight tiles, and as many K splits (one cluster, at most 8) as keep every
// SM streaming weights. Returns false when the tile kernel is the better fit.
struct SplitPlan {
    int bn, splits, kps, a_rows;
    fl::SplitGeom geom;
};

// Ring of the split-K kernel for a tile width, activation box height and
// cluster size: the two-CTAs-per-SM budget when it holds at least four
// stages and the reduction exchange, else the one-CTA budget. Returns false
// if neither holds the exchange.
template <int BN, bool DUAL>
bool split_geom_bn(int a_rows, int splits, fl::SplitGeom* g) {
    using C = fl::SplitCfg<BN, DUAL>;
    const int stage = a_rows * 128 + C::STAGE_B_BYTES;
    const int xbytes = C::xchg_bytes(splits, a_rows);
    int stages = std::min(C::MAX_STAGES, C::RING_SMALL / stage);
    if (stages < 4 || xbytes > stages * stage) stages = std::min(C::MAX_STAGES, C::RING_LARGE / stage);
    if (xbytes > stages * stage) return false;
    g->stages = stages;
    g->stage_bytes = stage;
    g->smem_bytes = C::smem_bytes(stages, stage);
    return true;
}

bool split_geom(int bn, bool dual, int a_rows, int splits, fl::SplitGeom* g) {
    if (dual) return bn == 128 ? split_geom_bn<128, true>(a_rows, splits, g) : split_geom_bn<64, true>(a_rows, splits, g);
    return bn == 128 ? split_geom_bn<128, false>(a_rows, splits, g) : split_geom_bn<64, false>(a_rows, splits, g);
}

int max_clusters(int dt, int bn, int pro, bool dual, int splits, int a_rows, int smem) {
    // cached per (dtype, width, prologue, dual, cluster size, box height); single device assumed per process slot
    static std::atomic<int> cache[2][2][4][2][9][8];
    const int bi = bn == 128 ? 1 : 0;
    const int ai = (a_rows / 16 - 1) & 7;
    int v = cache[dt][bi][pro][dual ? 1 : 0][splits][ai].load();
    if (v != 0) return v;
    if (dual) {
        if (pro == fl::PRO_RMS) {
            if (bn == 64) v = dt == 0 ? fl::splitk_max_clusters<0, 64, fl::PRO_RMS, true>(splits, smem)
                                      : fl::splitk_max_clusters<1, 64, fl::PRO_RMS, true>(splits, smem);
            else v = dt == 0 ? fl::splitk_max_clusters<0, 128, fl::PRO_RMS, true>(splits, smem)
                             : fl::splitk_max_clusters<1, 128, fl::PRO_RMS, true>(splits, smem);
        }
        if (v <= 0) v = -1;
        cache[dt][bi][pro][1][splits][ai] = v;
        return v;
    }
#define FL_Q(DT, BN, PRO) \
    if (dt == DT && bn == BN && pro == PRO) v = fl::splitk_max_clusters<DT, BN, PRO>(splits, smem);
    FL_Q(0, 64, 0) FL_Q(0, 64, 1) FL_Q(0, 64, 2) FL_Q(0, 64, 3) FL_Q(0, 128, 0) FL_Q(0, 128, 1) FL_Q(0, 128, 2)
    FL_Q(0, 128, 3) FL_Q(1, 64, 0) FL_Q(1, 64, 1) FL_Q(1, 64, 2) FL_Q(1, 64, 3) FL_Q(1, 128, 0) FL_Q(1, 128, 1)
    FL_Q(1, 128, 2) FL_Q(1, 128, 3)
#undef FL_Q
    if (v <= 0) v = -1;
    cache[dt][bi][pro][0][splits][ai] = v;
    return v;
}

// dual: the SwiGLU gate/up form (two weights, SwiGLU epilogue), taken for
// decode row counts, where the CTA-pair and tile kernels would run mostly
// empty 256- or 128-row MMAs over the whole K range.
bool plan_splitk(int dt, int pro, bool dual, int M, const Outs& outs, int K, int sms, SplitPlan* plan) {
    const int variant = g_opt_variant.load();
    if (variant == 1 || variant == 3) return false;
    const int nk = (K + fl::kBK - 1) / fl::kBK;
    const int mb = (M + fl::kBM - 1) / fl::kBM;
    // 128-wide weight tiles stage more bytes per pipeline slot (more bytes in
    // flight per SM); 64-wide ones give twice the CTAs. Prefer 128 unless it
    // leaves a quarter of the CTAs unused; past one 128-row block, where the
    // step is no longer a pure weight stream, take 64 on a tie if it still
    // splits K: the same CTAs with half the K split exchange half as much
    // (512 x 1024 x 1024: 7.2 against 8.3 us), while no split at all leaves
    // each CTA the whole K loop (512 x 2048 x 2048: 17.9 against 13.1 us).
    auto ctas_for = [&](int b) {
        const long long tl = mb * nblocks(outs, b);
        long long sp = sms / (tl > 0 ? tl : 1);
        if (sp > 8) sp = 8;
        while (sp > 1 && nk / sp < 2) --sp;
        return tl * (sp < 1 ? 1 : sp);
    };
    const int forced_bn = g_opt_tile_n.load();
    const long long c128 = ctas_for(128), c64 = ctas_for(64);
    const bool split64 = c64 >= 2ll * mb * nblocks(outs, 64);
    const int bn = forced_bn == 128 ? 128
                   : forced_bn == 256 ? 64
                   : (mb > 1 && split64 ? (c128 > c64 ? 128 : 64) : (c128 * 4 >= c64 * 3 ? 128 : 64));
    const long long tiles = mb * nblocks(outs, bn);
    // gate/up: up to 64 rows (at 128 rows the CTA-pair kernel measured faster:
    // 78 against 91 us for the 4096 x 11008 bf16 block)
    if (dual && (M > kDualSplitRows || pro != fl::PRO_RMS)) return false;
    if (variant == 0 && !dual) {
        // the tile kernel fills at least half the SMs: it reuses each staged
        // tile across the whole K loop and needs no reduction
        if ((long long)mb * nblocks(outs, 128) * 2 > sms || nk < 4) return false;
    }
    int splits = g_opt_split_k.load();
    if (splits <= 0) {
        splits = (int)(sms / (tiles > 0 ? tiles : 1));
        if (splits > 8) splits = 8;
        if (splits < 1) splits = 1;
        while (splits > 1 && nk / splits < 2) --splits;  // at least two K blocks per split
    }
    if (splits > nk) splits = nk;
    if (splits < 1) splits = 1;
    const int a_rows = M >= fl::kBM ? fl::kBM : (M + 15) / 16 * 16;
    // every cluster of the grid resident at once (one wave): the cluster shape
    // limits how many fit on the GPCs
    fl::SplitGeom geom;
    for (;; --splits) {
        if (splits < 1) return false;
        if (!split_geom(bn, dual, a_rows, splits, &geom)) continue;
        if (splits == 1) break;
        const int mc = max_clusters(dt, bn, pro, dual, splits, a_rows, geom.smem_bytes);
        if (mc < 0 || tiles <= mc) break;
    }
    const int kps = (nk + splits - 1) / splits;
    plan->bn = bn;
    plan->kps = kps;
    plan->splits = (nk + kps - 1) / kps;  // every split gets at least one K block
    plan->a_rows = a_rows;
    if (!split_geom(bn, dual, a_rows, plan->splits, &plan->geom)) return false;
    return true;
}

int pair_max(int dt, int bn, int pro, int ks) {
    // resident clusters (of 2 * ks CTAs) of each pair-kernel instance, cached
    static std::atomic<int> cache[2][3][4];
    const int ci = ks == 2 ? 2 : (bn == 256 ? 1 : 0);
    int v = cache[dt][ci][pro].load();
    if (v != 0) return v;
#define FL_Q(DT, BN, PRO, KS) \
    if (dt == DT && bn == BN && pro == PRO && ks == KS) v = fl::pair_max_clusters<DT, BN, PRO, KS>();
    FL_Q(0, 128, 0, 1) FL_Q(0, 128, 1, 1) FL_Q(0, 128, 2, 1) FL_Q(0, 128, 3, 1)
    FL_Q(0, 256, 0, 1) FL_Q(0, 256, 1, 1) FL_Q(0, 256, 2, 1) FL_Q(0, 256, 3, 1)
    FL_Q(1, 128, 0, 1) FL_Q(1, 128, 1, 1) FL_Q(1, 128, 2, 1) FL_Q(1, 128, 3, 1)
    FL_Q(1, 256, 0, 1) FL_Q(1, 256, 1, 1) FL_Q(1, 256, 2, 1) FL_Q(1, 256, 3, 1)
    FL_Q(0, 256, 0, 2) FL_Q(0, 256, 1, 2) FL_Q(0, 256, 2, 2) FL_Q(0, 256, 3, 2)
    FL_Q(1, 256, 0, 2) FL_Q(1, 256, 1, 2) FL_Q(1, 256, 2, 2) FL_Q(1, 256, 3, 2)
#undef FL_Q
    if (v <= 0) v = -1;
    cache[dt][ci][pro] = v;
    return v;
}

cudaError_t dispatch_pair(int dt, int bn, int pro, int ks, bool dual, const GemmParamsMulti& p, int grid,
                          cudaStream_t s) {
    if (p.n_out > 1) {
#define FL_CASE(DT, PRO, KS) \
        if (dt == DT && bn == 256 && pro == PRO && ks == KS && !dual)   \
            return fl::launch_pair<DT, 256, PRO, KS, false, true>(p, grid, s);
        FL_CASE(0, 1, 1) FL_CASE(0, 2, 1) FL_CASE(0, 1, 2) FL_CASE(0, 2, 2)
        FL_CASE(1, 1, 1) FL_CASE(1, 2, 1) FL_CASE(1, 1, 2) FL_CASE(1, 2, 2)
#undef FL_CASE
        return cudaErrorInvalidValue;
    }
    if (dual) {
        if (bn != 256 || pro != fl::PRO_RMS || ks != 1) return cudaErrorInvalidValue;
        return dt == 0 ? fl::launch_pair<0, 256, fl::PRO_RMS, 1, true>(p, grid, s)
                       : fl::launch_pair<1, 256, fl::PRO_RMS, 1, true>(p, grid, s);
    }
#define FL_CASE(DT, BN, PRO, KS) \
    if (dt == DT && bn == BN && pro == PRO && ks == KS) return fl::launch_pair<DT, BN, PRO, KS, false>(p, grid, s);
    FL_CASE(0, 128, 0, 1) FL_CASE(0, 128, 1, 1) FL_CASE(0, 128, 2, 1) FL_CASE(0, 128, 3, 1)
    FL_CASE(0, 256, 0, 1) FL_CASE(0, 256, 1, 1) FL_CASE(0, 256, 2, 1) FL_CASE(0, 256, 3, 1)
    FL_CASE(1, 128, 0, 1) FL_CASE(1, 128, 1, 1) FL_CASE(1, 128, 2, 1) FL_CASE(1, 128, 3, 1)
    FL_CASE(1, 256, 0, 1) FL_CASE(1, 256, 1, 1) FL_CASE(1, 256, 2, 1) FL_CASE(1, 256, 3, 1)
    FL_CASE(0, 256, 0, 2) FL_CASE(0, 256, 1, 2) FL_CASE(0, 256, 2, 2) FL_CASE(0, 256, 3, 2)
    FL_CASE(1, 256, 0, 2) FL_CASE(1, 256, 1, 2) FL_CASE(1, 256, 2, 2) FL_CASE(1, 256, 3, 2)
#undef FL_CASE
    return cudaErrorInvalidValue;
}

struct PairPlan {
    int bn, ks, clusters;
};

int choose_bn(int M, const Outs& outs, bool dual, int sms);

// The CTA-pair kernel, when its 256-wide tiles keep 80 % of the resident pairs
// busy: directly, or with each tile's K range split over two pairs (a cluster
// of four) when there are half as many tiles. A 128-wide pair tile moves as
// many shared-memory bytes per MMA as the single-CTA 128 x 256 tile and
// measures no faster, so it is used only when forced (FL_OPT_VARIANT = 3 with
// FL_OPT_TILE_N = 128; FL_OPT_SPLIT_K = 2 forces the K split).
bool use_pair(int dt, int pro, int M, const Outs& outs, int K, PairPlan* plan, bool dual, int sms) {
    const int variant = g_opt_variant.load();
    if (variant == 1 || variant == 2) return false;
    if (dual) {
        // SwiGLU gate/up: 128 output columns per 256 x 256 pair tile (Wg and Wu
        // stacked); no K split, no 128-wide variant. Decode row counts (one
        // 128-row block) take the split-K form instead.
        if (pro != fl::PRO_RMS) return false;
        if (variant != 3 && M <= kDualSplitRows) return false;
        const long long tiles = (long long)((M + 255) / 256) * nblocks(outs, 128);
        const int maxp = pair_max(dt, 256, pro, 1);
        if (maxp <= 0) return false;
        if (variant != 3 && tiles * 5 < (long long)maxp * 4) return false;
        *plan = PairPlan{256, 1, (int)(tiles < maxp ? tiles : maxp)};
        return true;
    }
    const int forced_bn = g_opt_tile_n.load();
    const int forced_split = g_opt_split_k.load();
    const long long mp = (M + 255) / 256;
    const long long t256 = mp * nblocks(outs, 256), t128 = mp * nblocks(outs, 128);
    const int nk = (K + fl::kBK - 1) / fl::kBK;
    if (variant == 3 && forced_bn == 128 && outs.n == 1) {
        const int maxp = pair_max(dt, 128, pro, 1);
        if (maxp <= 0) return false;
        *plan = PairPlan{128, 1, (int)(t128 < maxp ? t128 : maxp)};
        return true;
    }
    const int maxp = pair_max(dt, 256, pro, 1);
    if (maxp <= 0) return false;
    const bool fills = t256 * 5 >= (long long)maxp * 4;
    const int maxq = pair_max(dt, 256, pro, 2);
    const bool split_fits = maxq > 0 && t256 <= maxq && nk >= 8;
    const bool split = forced_split == 2 ? split_fits
                                         : (!fills && split_fits && t256 * 2 * 5 >= (long long)maxp * 4);
    if (split) {
        *plan = PairPlan{256, 2, (int)t256};
        return true;
    }
    // too few tiles to fill the pairs, but the pair tiles still cover as many
    // SMs as the 1-CTA kernel's tiles would: the pair moves fewer shared-memory
    // bytes per MMA (QKV 4096 + 1024 + 1024 at M = 512: 28.6 against 36.0 us)
    // (Not where the split-K kernel takes the shape: few row blocks, where
    // one K-split cluster per 128-row tile streams the weight once.)
    long long tile_ctas = 0;
    const long long mb128 = (M + fl::kBM - 1) / fl::kBM;
    if (variant == 0 && !fills && (mb128 * nblocks(outs, 128) * 2 > sms || nk < 4)) {
        const long long t1 = (long long)((M + fl::kBM - 1) / fl::kBM) * nblocks(outs, choose_bn(M, outs, false, sms));
        tile_ctas = t1 < sms ? t1 : sms;
    }
    const bool covers = tile_ctas > 0 && t256 * 2 >= tile_ctas && t256 <= maxp;
    if (variant != 3 && !fills && !covers) return false;
    *plan = PairPlan{256, 1, (int)(t256 < maxp ? t256 : maxp)};
    return true;
}

// Fields every launch shares.
void fill_common(GemmParamsMulti& p, const void* A, const void* residual, const void* gamma, const void* beta,
                 const void* ln_stats, int M, int K, float eps, DeviceInfo* di) {
    p.ln_stats = ln_stats;
    p.residual = residual;
    p.gamma = gamma;
    p.beta = beta;
    p.a_ptr = A;
    p.status = di->status;
    p.timeout_ns = (unsigned long long)g_opt_timeout_ms.load() * 1000000ull;
    p.M = M;
    p.K = K;
    p.num_k_blocks = (K + fl::kBK - 1) / fl::kBK;
    p.eps = eps;
    p.pdl = g_opt_pdl.load();
}

fl_status encode_prologue(GemmParamsMulti& p, int dt, int pro, const void* gamma, const void* beta, int K) {
    fl_status st;
    if (pro != fl::PRO_NONE && (st = encode_2d(&p.tmGamma, dt, gamma, K, 1, fl::kBK, 1, false)) != FL_OK) return st;
    if (pro == fl::PRO_LN && beta != nullptr && (st = encode_2d(&p.tmBeta, dt, beta, K, 1, fl::kBK, 1, false)) != FL_OK)
        return st;
    return FL_OK;
}

// A launch whose parameters are built: the kernel family, its template
// arguments, the grid and the parameter block (tensor maps encoded).
enum LaunchPath : int { PATH_TILE = 0, PATH_SPLITK = 1, PATH_PAIR = 2 };
struct Prepared {
    int path, dt, pro, bn, ks, splits, grid;
    bool dual;
    GemmParamsMulti p;
};

fl_status prepare_pair(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2,
                       const void* residual, const void* gamma, const void* beta, int M, int K, float eps,
                       const PairPlan& plan, DeviceInfo* di, Prepared* out) {
    const int bn = plan.bn;
    GemmParamsMulti& p = out->p;
    memset(&p, 0, sizeof(p));
    fill_common(p, A, residual, gamma, beta, nullptr, M, K, eps, di);
    fl_status st;
    if ((st = encode_2d(&p.tmA, dt, A, K, M, fl::kBK, fl::kBM)) != FL_OK) return st;
    // output columns of a tile: the pair's 256-row weight tile holds bn
    // columns of one weight, or (gate/up) bn / 2 columns of Wg over Wu
    if ((st = fill_outputs(p, dt, outs, M, K, dual ? bn / 2 : bn, bn / 2)) != FL_OK) return st;
    if (dual && (st = encode_2d(&p.tmB2, dt, W2, K, outs.o[0].N, fl::kBK, bn / 2)) != FL_OK) return st;
    if ((st = encode_prologue(p, dt, pro, gamma, beta, K)) != FL_OK) return st;
    p.num_m_blocks = (M + 255) / 256;  // row blocks of a pair tile
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.splits = plan.ks;
    p.kps = (p.num_k_blocks + plan.ks - 1) / plan.ks;
    out->path = PATH_PAIR;
    out->bn = bn;
    out->ks = plan.ks;
    out->grid = 2 * plan.ks * plan.clusters;
    return FL_OK;
}

// CTA tile width. A wider tile halves the activation re-reads and the shared
// memory traffic per MMA, but fewer tiles may leave SMs idle: take the width
// whose whole waves of CTAs cost least.
int choose_bn(int M, const Outs& outs, bool dual, int sms) {
    if (dual) return 128;
    const int forced = g_opt_tile_n.load();
    if (forced == 128 || forced == 256) return forced;
    const long long mb = (M + fl::kBM - 1) / fl::kBM;
    const long long t256 = mb * nblocks(outs, 256), t128 = mb * nblocks(outs, 128);
    const long long w256 = (t256 + sms - 1) / sms, w128 = (t128 + sms - 1) / sms;
    // relative cost of one wave: a 128-wide tile does half the MMA work of a
    // 256-wide one but is less efficient per flop
    const double c256 = (double)w256 * 2.0, c128 = (double)w128 * 1.15;
    return c256 <= c128 ? 256 : 128;
}

fl_status prepare_splitk(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2,
                         const void* residual, const void* gamma, const void* beta, int M, int K, float eps,
                         const SplitPlan& plan, DeviceInfo* di, Prepared* out) {
    GemmParamsMulti& p = out->p;
    memset(&p, 0, sizeof(p));
    fill_common(p, A, residual, gamma, beta, nullptr, M, K, eps, di);
    const int a_rows = plan.a_rows;
    fl_status st;
    if ((st = encode_2d(&p.tmA, dt, A, K, M, fl::kBK, a_rows)) != FL_OK) return st;
    if ((st = fill_outputs(p, dt, outs, M, K, plan.bn, plan.bn)) != FL_OK) return st;
    if (dual && (st = encode_2d(&p.tmB2, dt, W2, K, outs.o[0].N, fl::kBK, plan.bn)) != FL_OK) return st;
    if ((st = encode_prologue(p, dt, pro, gamma, beta, K)) != FL_OK) return st;
    p.num_m_blocks = (M + fl::kBM - 1) / fl::kBM;
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.splits = plan.splits;
    p.kps = plan.kps;
    p.a_rows = a_rows;
    p.s_stages = plan.geom.stages;
    p.s_stage_bytes = plan.geom.stage_bytes;
    p.w_preload = g_opt_preload.load();
    p.s_one_per_sm = plan.geom.smem_bytes * 2 + 2048 > 228 * 1024;  // one CTA per SM
    {
        const int nch = plan.bn / 8, s = plan.splits;
        for (int d = 0; d <= s; ++d) p.xc_c0[d] = (unsigned char)(d * nch / s);
        for (int d = 0; d < s; ++d)
            for (int ch = p.xc_c0[d]; ch < p.xc_c0[d + 1]; ++ch) {
                p.xc_owner[ch] = (unsigned char)d;
                p.xc_pos[ch] = (unsigned char)(ch - p.xc_c0[d]);
            }
        p.xc_stride = (nch + s - 1) / s * 8 * (dual ? 2 : 1) + 4;  // SplitCfg::xchg_stride
        p.inv_k = 1.0f / (float)K;
    }
    out->path = PATH_SPLITK;
    out->bn = plan.bn;
    out->splits = plan.splits;
    out->grid = p.num_tiles * plan.splits;
    return FL_OK;
}

fl_status prepare_kernels(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2,
                          const void* residual, const void* gamma, const void* beta, int M, int K, float eps,
                          DeviceInfo* di, Prepared* out) {
    out->dt = dt;
    out->pro = pro;
    out->dual = dual;
    out->ks = out->splits = 1;
    PairPlan pplan;
    if (use_pair(dt, pro, M, outs, K, &pplan, dual, di->sms))
        return prepare_pair(dt, pro, dual, A, outs, W2, residual, gamma, beta, M, K, eps, pplan, di, out);
    SplitPlan plan;
    if (plan_splitk(dt, pro, dual, M, outs, K, di->sms, &plan))
        return prepare_splitk(dt, pro, dual, A, outs, W2, residual, gamma, beta, M, K, eps, plan, di, out);
    const int bn = choose_bn(M, outs, dual, di->sms);
    GemmParamsMulti& p = out->p;
    memset(&p, 0, sizeof(p));
    fill_common(p, A, residual, gamma, beta, nullptr, M, K, eps, di);
    fl_status st;
    if ((st = encode_2d(&p.tmA, dt, A, K, M, fl::kBK, fl::kBM)) != FL_OK) return st;
    if ((st = fill_outputs(p, dt, outs, M, K, bn, bn)) != FL_OK) return st;
    if (dual && (st = encode_2d(&p.tmB2, dt, W2, K, outs.o[0].N, fl::kBK, bn)) != FL_OK) return st;
    if ((st = encode_prologue(p, dt, pro, gamma, beta, K)) != FL_OK) return st;
    p.num_m_blocks = (M + fl::kBM - 1) / fl::kBM;
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    out->path = PATH_TILE;
    out->bn = bn;
    out->grid = p.num_tiles < di->sms ? p.num_tiles : di->sms;
    return FL_OK;
}

// Kernels launched (issued to a stream, or recorded into a captured graph)
// since the library was loaded, counted on the host after each successful
// launch call.
std::atomic<long long> g_kernel_launches{0};

void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

fl_status launch_prepared(const Prepared& L, cudaStream_t stream) {
    cudaError_t e;
    const char* what;
    if (L.path == PATH_PAIR) {
        e = dispatch_pair(L.dt, L.bn, L.pro, L.ks, L.dual, L.p, L.grid, stream);
        what = "pair kernel launch failed";
    } else if (L.path == PATH_SPLITK) {
        e = dispatch_splitk(L.dt, L.bn, L.pro, L.dual, L.p, L.grid, L.splits, stream);
        what = "split-K kernel launch failed";
    } else {
        e = dispatch_tile(L.dt, L.bn, L.pro, L.dual, L.p, L.grid, stream);
        what = "kernel launch failed";
    }
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    count_launch();
    return ok();
}

// ---------------------------------------------------------------------------
// launch cache
// ---------------------------------------------------------------------------
// A call repeated with the same pointers, sizes and options (every step of a
// decode loop, every layer of a model) gets the same kernel choice and the
// same tensor maps: those are kept per argument set, so a repeated call only
// validates, looks up and launches. Key: everything the preparation reads,
// compared byte for byte (the key is zeroed before it is filled, so padding
// compares equal).
struct CallKey {
    int device, dt, pro, dual, M, K, n;
    uint32_t eps_bits;
    const void *A, *W2, *residual, *gamma, *beta;
    OutDesc o[fl::kMaxOut];
    int opt_tile_n, opt_variant, opt_split_k, opt_pdl, opt_preload, opt_timeout_ms;
};

constexpr int kCacheSlots = 64;
struct CacheSlot {
    bool used = false;
    CallKey key;
    Prepared prep;
};
CacheSlot g_cache[kCacheSlots];
std::mutex g_cache_mu;
std::atomic<long long> g_cache_hits{0}, g_cache_misses{0};

uint64_t hash_bytes(const void* data, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(data);
    uint64_t h = 1469598103934665603ull;  // FNV-1a
    for (size_t i = 0; i < n; ++i) {
        h ^= b[i];
        h *= 1099511628211ull;
    }
    return h;
}

fl_status run_kernels(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2,
                      const void* residual, const void* gamma, const void* beta, const void* ln_stats, int M, int K,
                      float eps, DeviceInfo* di, int device, cudaStream_t stream) {
    CallKey key;
    memset(&key, 0, sizeof(key));
    key.device = device;
    key.dt = dt;
    key.pro = pro;
    key.dual = dual;
    key.M = M;
    key.K = K;
    key.n = outs.n;
    memcpy(&key.eps_bits, &eps, sizeof(float));
    key.A = A;
    key.W2 = W2;
    key.residual = residual;
    key.gamma = gamma;
    key.beta = beta;
    for (int i = 0; i < outs.n; ++i) key.o[i] = outs.o[i];
    key.opt_tile_n = g_opt_tile_n.load();
    key.opt_variant = g_opt_variant.load();
    key.opt_split_k = g_opt_split_k.load();
    key.opt_pdl = g_opt_pdl.load();
    key.opt_preload = g_opt_preload.load();
    key.opt_timeout_ms = g_opt_timeout_ms.load();
    CacheSlot& slot = g_cache[hash_bytes(&key, sizeof(key)) % kCacheSlots];
    // one prepared launch per call on the stack (about 2 KB)
    Prepared prep;
    bool hit = false;
    const bool use_cache = g_opt_cache.load() != 0;
    if (use_cache) {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        if (slot.used && memcmp(&slot.key, &key, sizeof(key)) == 0) {
            prep = slot.prep;
            hit = true;
        }
    }
    if (hit) {
        g_cache_hits.fetch_add(1, std::memory_order_relaxed);
    } else {
        g_cache_misses.fetch_add(1, std::memory_order_relaxed);
        fl_status st = prepare_kernels(dt, pro, dual, A, outs, W2, residual, gamma, beta, M, K, eps, di, &prep);
        if (st != FL_OK) return st;
        if (use_cache) {
            std::lock_guard<std::mutex> lk(g_cache_mu);
            slot.key = key;
            slot.prep = prep;
            slot.used = true;
        }
    }
    prep.p.ln_stats = ln_stats;  // per-call scratch, not part of the key
    prep.p.status = stream_status(di, stream);
#ifdef FL_TRACE
    if (const char* tp = getenv("FL_TRACE_PTR"))
        prep.p.trace = reinterpret_cast<unsigned long long*>(strtoull(tp, nullptr, 10));
#endif
    return launch_prepared(prep, stream);
}

// One fused call. LayerNorm first computes the row statistics (8 bytes per
// row of stream-ordered scratch from the library pool, freed on the stream
// right after the GEMM kernel that reads them), once for all outputs.
// Decode row counts go to the weight-streaming decode kernel (8-row units per
// CTA, warp-level MMAs, no reduction across CTAs); FL_OPT_VARIANT = 4 forces
// it where it fits.
// Automatic choice: up to 4 rows; up to 8 rows while K <= 2048; and 5 to 8
// rows at larger K for plain or RMSNorm / input-bias prologues with one or
// several outputs (4096 x 4096 at M = 5 / 6 / 8: 9.6 / 9.8 / 10.2 against
// 10.1 us on the split-K tcgen05 kernel; QKV at M = 8: 13.4 against 14.8),
// but not for the SwiGLU gate/up pair (62 against 55 us at M = 6 and 8,
// 4096 / 11008) nor LayerNorm (14.7 against 13.3 us at M = 8).
bool use_gemv(int M, int K, int pro, bool dual) {
    const int variant = g_opt_variant.load();
    if (variant != 0 && variant != 4) return false;
    if (M > fl::kGemvMaxRows || fl::gemv_smem_bytes(M, K, pro) > fl::kGemvSmemMax) return false;
    return variant == 4 || M <= 4 || K <= 2048 || (!dual && pro != fl::PRO_LN);
}

// dual: the SwiGLU gate/up pair (outs.o[0].W = Wg, W2 = Wu, out = h).
fl_status run_gemv(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2, const void* residual,
                   const void* gamma, const void* beta, int M, int K, float eps, DeviceInfo* di,
                   cudaStream_t stream) {
    fl::GemvParams g;
    memset(&g, 0, sizeof(g));
    g.x = static_cast<const uint16_t*>(A);
    g.gamma = static_cast<const uint16_t*>(gamma);
    g.beta = static_cast<const uint16_t*>(beta);
    g.n_out = outs.n;
    int rows = 0;
    for (int i = 0; i < outs.n; ++i) {
        g.W[i] = static_cast<const uint16_t*>(outs.o[i].W);
        g.bias[i] = static_cast<const uint16_t*>(outs.o[i].bias);
        g.out[i] = static_cast<uint16_t*>(outs.o[i].out);
        g.N[i] = outs.o[i].N;
        g.act[i] = outs.o[i].act;
        g.row0[i] = rows;
        rows += outs.o[i].N;
    }
    for (int i = outs.n; i <= 4; ++i) g.row0[i] = rows;
    if (dual) g.W[1] = static_cast<const uint16_t*>(W2);
    g.residual = static_cast<const uint16_t*>(residual);
    g.M = M;
    g.K = K;
    g.eps = eps;
#ifdef FL_TRACE
    if (const char* tp = getenv("FL_TRACE_PTR"))
        g.trace = reinterpret_cast<unsigned long long*>(strtoull(tp, nullptr, 10));
#endif
    const cudaError_t e = fl::launch_gemv(dt, pro, dual, g, di->sms, g_opt_pdl.load(), stream);
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "decode kernel launch failed: %s", cudaGetErrorString(e));
    count_launch();
    return ok();
}

fl_status run_tile(int dt, int pro, bool dual, const void* A, const Outs& outs, const void* W2,
                   const void* residual, const void* gamma, const void* beta, int M, int K, float eps,
                   cudaStream_t stream) {
    DeviceInfo* di = nullptr;
    fl_status st = device_info(&di);
    if (st != FL_OK) return st;
    // (the decode kernel computes its few rows' LayerNorm statistics itself)
    if (use_gemv(M, K, pro, dual) && (!dual || pro == fl::PRO_RMS))
        return run_gemv(dt, pro, dual, A, outs, W2, residual, gamma, beta, M, K, eps, di, stream);
    void* stats = nullptr;
    if (pro == fl::PRO_LN) {
        cudaError_t e = cudaMallocFromPoolAsync(&stats, (size_t)M * 8, di->pool, stream);
        if (e != cudaSuccess) return fail(FL_ERR_CUDA, "LayerNorm statistics scratch: %s", cudaGetErrorString(e));
        e = fl::launch_ln_stats(dt, A, M, K, eps, stats, g_opt_pdl.load(), di->sms, stream);
        if (e != cudaSuccess) {
            cudaFreeAsync(stats, stream);
            return fail(FL_ERR_CUDA, "LayerNorm statistics kernel launch failed: %s", cudaGetErrorString(e));
        }
        count_launch();
    }
    st = run_kernels(dt, pro, dual, A, outs, W2, residual, gamma, beta, stats, M, K, eps, di, device_index(), stream);
    if (stats != nullptr) cudaFreeAsync(stats, stream);
    return st;
}

// Common shape checks of one GEMM [M,K] x [N,K]^T.
fl_status check_shape(const char* what, long long M, long long N, long long K) {
    if (M < 1 || N < 1 || K < 1) return fail(FL_ERR_INVALID_ARG, "%s: sizes must be positive (M=%lld N=%lld K=%lld)", what, M, N, K);
    if (N % 8 != 0 || K % 8 != 0)
        return fail(FL_ERR_ALIGNMENT, "%s: N and K must be multiples of 8 (N=%lld K=%lld)", what, N, K);
    const long long mb = (M + 127) / 128, nb = (N + 63) / 64;
    if (mb * nb > INT_MAX / 2) return fail(FL_ERR_UNSUPPORTED, "%s: too many output tiles", what);
    return FL_OK;
}

fl_status check_ptr(const char* name, const void* p, bool required) {
    if (p == nullptr) {
        if (required) return fail(FL_ERR_INVALID_ARG, "%s must not be null", name);
        return FL_OK;
    }
    if (!aligned16(p)) return fail(FL_ERR_ALIGNMENT, "%s must be 16-byte aligned", name);
    return FL_OK;
}

bool valid_dtype(int dt) { return dt == FL_F16 || dt == FL_BF16; }

}  // namespace

int fl::set_last_error(int status, const char* message) { return fail((fl_status)status, "%s", message); }

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* fl_last_error(void) { return tls_err; }

const char* fl_version(void) { return "libfusedlin 0.1 (sm_103a, tcgen05 + TMA)"; }

fl_status fl_set_option(fl_option key, int value) {
    switch (key) {
        case FL_OPT_TILE_N:
            if (value != 0 && value != 128 && value != 256) return fail(FL_ERR_INVALID_ARG, "tile width must be 0, 128 or 256");
            g_opt_tile_n = value;
            return ok();
        case FL_OPT_VARIANT:
            if (value < 0 || value > 4) return fail(FL_ERR_INVALID_ARG, "variant must be 0..4");
            g_opt_variant = value;
            return ok();
        case FL_OPT_TIMEOUT_MS:
            if (value < 1 || value > 600000) return fail(FL_ERR_INVALID_ARG, "timeout must be 1..600000 ms");
            g_opt_timeout_ms = value;
            return ok();
        case FL_OPT_SPLIT_K:
            if (value < 0 || value > 8) return fail(FL_ERR_INVALID_ARG, "split must be 0..8");
            g_opt_split_k = value;
            return ok();
        case FL_OPT_PDL:
            if (value < 0 || value > 1) return fail(FL_ERR_INVALID_ARG, "pdl must be 0 or 1");
            g_opt_pdl = value;
            return ok();
        case FL_OPT_WEIGHT_PRELOAD:
            if (value < 0 || value > 1) return fail(FL_ERR_INVALID_ARG, "weight preload must be 0 or 1");
            g_opt_preload = value;
            return ok();
        case FL_OPT_LAUNCH_CACHE:
            if (value < 0 || value > 1) return fail(FL_ERR_INVALID_ARG, "launch cache must be 0 or 1");
            g_opt_cache = value;
            return ok();
        default:
            return fail(FL_ERR_INVALID_ARG, "unknown option %d", (int)key);
    }
}

fl_status fl_gemm_epilogue(const void* A, const void* W, const void* bias, const void* residual, void* out, int M,
                           int N, int K, fl_pattern pattern, fl_dtype dtype, void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if ((int)pattern < 0 || (int)pattern > FL_RMSNORM_GEMM) return fail(FL_ERR_INVALID_ARG, "bad pattern %d", (int)pattern);
    if (pattern == FL_LAYERNORM_GEMM || pattern == FL_RMSNORM_GEMM)
        return fail(FL_ERR_INVALID_ARG, "norm patterns take gamma/eps: call fl_norm_gemm");
    const bool uses_bias = pattern <= FL_GEMM_BIAS_RESIDUAL;
    const bool uses_res = pattern == FL_GEMM_BIAS_RESIDUAL;
    int act = fl::ACT_NONE;
    if (pattern == FL_GEMM_BIAS_GELU || pattern == FL_GEMM_GELU) act = fl::ACT_GELU;
    if (pattern == FL_GEMM_BIAS_SILU || pattern == FL_GEMM_SILU) act = fl::ACT_SILU;
    if (pattern == FL_GEMM_BIAS_RELU) act = fl::ACT_RELU;
    fl_status st;
    if ((st = check_shape("fl_gemm_epilogue", M, N, K)) != FL_OK) return st;
    if ((st = check_ptr("A", A, true)) != FL_OK) return st;
    if ((st = check_ptr("W", W, true)) != FL_OK) return st;
    if ((st = check_ptr("out", out, true)) != FL_OK) return st;
    if ((st = check_ptr("bias", uses_bias ? bias : nullptr, uses_bias)) != FL_OK) return st;
    if ((st = check_ptr("residual", uses_res ? residual : nullptr, uses_res)) != FL_OK) return st;
    const size_t ob = (size_t)M * N * 2;
    if (overlap(out, ob, A, (size_t)M * K * 2) || overlap(out, ob, W, (size_t)N * K * 2) ||
        (uses_bias && overlap(out, ob, bias, (size_t)N * 2)))
        return fail(FL_ERR_INVALID_ARG, "out overlaps an input");
    if (uses_res && residual != out && overlap(out, ob, residual, ob))
        return fail(FL_ERR_INVALID_ARG, "out may alias residual only exactly");
    return run_tile(dtype, fl::PRO_NONE, false, A, single_out(W, uses_bias ? bias : nullptr, out, N, act), nullptr,
                    uses_res ? residual : nullptr, nullptr, nullptr, M, K, 0.f, static_cast<cudaStream_t>(stream));
}

fl_status fl_norm_gemm(const void* x, const void* gamma, const void* beta, const void* W, const void* bias, void* out,
                       int M, int N, int K, float eps, fl_norm_kind norm_kind, fl_act act, fl_dtype dtype,
                       void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if (norm_kind != FL_NORM_RMS && norm_kind != FL_NORM_LAYER)
        return fail(FL_ERR_INVALID_ARG, "bad norm kind %d", (int)norm_kind);
    if ((int)act < 0 || (int)act > FL_ACT_RELU) return fail(FL_ERR_INVALID_ARG, "bad activation %d", (int)act);
    if (!(eps >= 0.0f) || eps > 1e30f) return fail(FL_ERR_INVALID_ARG, "eps must be finite and >= 0");
    fl_status st;
    if ((st = check_shape("fl_norm_gemm", M, N, K)) != FL_OK) return st;
    if ((st = check_ptr("x", x, true)) != FL_OK) return st;
    if ((st = check_ptr("gamma", gamma, true)) != FL_OK) return st;
    if ((st = check_ptr("W", W, true)) != FL_OK) return st;
    if ((st = check_ptr("out", out, true)) != FL_OK) return st;
    if ((st = check_ptr("bias", bias, false)) != FL_OK) return st;
    const void* b = norm_kind == FL_NORM_LAYER ? beta : nullptr;
    if ((st = check_ptr("beta", b, false)) != FL_OK) return st;
    const size_t ob = (size_t)M * N * 2;
    if (overlap(out, ob, x, (size_t)M * K * 2) || overlap(out, ob, W, (size_t)N * K * 2) ||
        overlap(out, ob, gamma, (size_t)K * 2) || overlap(out, ob, b, (size_t)K * 2) ||
        overlap(out, ob, bias, (size_t)N * 2))
        return fail(FL_ERR_INVALID_ARG, "out overlaps an input");
    const int pro = norm_kind == FL_NORM_RMS ? fl::PRO_RMS : fl::PRO_LN;
    return run_tile(dtype, pro, false, x, single_out(W, bias, out, N, (int)act), nullptr, nullptr, gamma, b, M, K, eps,
                    static_cast<cudaStream_t>(stream));
}

fl_status fl_norm_gemm_multi(const void* x, const void* gamma, const void* beta, int n_out, const void* const* W,
                             const void* const* bias, void* const* out, const int* N, const int* act, int M, int K,
                             float eps, fl_norm_kind norm_kind, fl_dtype dtype, void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if (norm_kind != FL_NORM_RMS && norm_kind != FL_NORM_LAYER)
        return fail(FL_ERR_INVALID_ARG, "bad norm kind %d", (int)norm_kind);
    if (n_out < 1 || n_out > FL_MAX_OUTPUTS || n_out > fl::kMaxOut)
        return fail(FL_ERR_INVALID_ARG, "n_out must be 1..%d, got %d", FL_MAX_OUTPUTS, n_out);
    if (W == nullptr || out == nullptr || N == nullptr)
        return fail(FL_ERR_INVALID_ARG, "W, out and N arrays must not be null");
    if (!(eps >= 0.0f) || eps > 1e30f) return fail(FL_ERR_INVALID_ARG, "eps must be finite and >= 0");
    fl_status st;
    if ((st = check_ptr("x", x, true)) != FL_OK) return st;
    if ((st = check_ptr("gamma", gamma, true)) != FL_OK) return st;
    const void* b = norm_kind == FL_NORM_LAYER ? beta : nullptr;
    if ((st = check_ptr("beta", b, false)) != FL_OK) return st;
    Outs outs;
    outs.n = n_out;
    for (int i = 0; i < n_out; ++i) {
        const int a = act != nullptr ? act[i] : FL_ACT_NONE;
        if (a < 0 || a > FL_ACT_RELU) return fail(FL_ERR_INVALID_ARG, "bad activation %d for output %d", a, i);
        if ((st = check_shape("fl_norm_gemm_multi", M, N[i], K)) != FL_OK) return st;
        if ((st = check_ptr("W[i]", W[i], true)) != FL_OK) return st;
        if ((st = check_ptr("out[i]", out[i], true)) != FL_OK) return st;
        const void* bi = bias != nullptr ? bias[i] : nullptr;
        if ((st = check_ptr("bias[i]", bi, false)) != FL_OK) return st;
        outs.o[i] = OutDesc{W[i], bi, out[i], N[i], a};
    }
    // every output overlaps no input and no other output
    for (int i = 0; i < n_out; ++i) {
        const size_t ob = (size_t)M * N[i] * 2;
        if (overlap(out[i], ob, x, (size_t)M * K * 2) || overlap(out[i], ob, gamma, (size_t)K * 2) ||
            overlap(out[i], ob, b, (size_t)K * 2))
            return fail(FL_ERR_INVALID_ARG, "out[%d] overlaps an input", i);
        for (int j = 0; j < n_out; ++j) {
            if (overlap(out[i], ob, outs.o[j].W, (size_t)N[j] * K * 2) ||
                overlap(out[i], ob, outs.o[j].bias, (size_t)N[j] * 2))
                return fail(FL_ERR_INVALID_ARG, "out[%d] overlaps an input", i);
            if (j != i && overlap(out[i], ob, out[j], (size_t)M * N[j] * 2))
                return fail(FL_ERR_INVALID_ARG, "out[%d] overlaps out[%d]", i, j);
        }
    }
    const int pro = norm_kind == FL_NORM_RMS ? fl::PRO_RMS : fl::PRO_LN;
    return run_tile(dtype, pro, false, x, outs, nullptr, nullptr, gamma, b, M, K, eps,
                    static_cast<cudaStream_t>(stream));
}

fl_status fl_input_bias_gemm(const void* A, const void* bias_in, const void* W, const void* bias, const void* residual,
                             void* out, int M, int N, int K, fl_act act, fl_dtype dtype, void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if ((int)act < 0 || (int)act > FL_ACT_RELU) return fail(FL_ERR_INVALID_ARG, "bad activation %d", (int)act);
    fl_status st;
    if ((st = check_shape("fl_input_bias_gemm", M, N, K)) != FL_OK) return st;
    if ((st = check_ptr("A", A, true)) != FL_OK) return st;
    if ((st = check_ptr("bias_in", bias_in, true)) != FL_OK) return st;
    if ((st = check_ptr("W", W, true)) != FL_OK) return st;
    if ((st = check_ptr("out", out, true)) != FL_OK) return st;
    if ((st = check_ptr("bias", bias, false)) != FL_OK) return st;
    if ((st = check_ptr("residual", residual, false)) != FL_OK) return st;
    const size_t ob = (size_t)M * N * 2;
    if (overlap(out, ob, A, (size_t)M * K * 2) || overlap(out, ob, W, (size_t)N * K * 2) ||
        overlap(out, ob, bias_in, (size_t)K * 2) || overlap(out, ob, bias, (size_t)N * 2))
        return fail(FL_ERR_INVALID_ARG, "out overlaps an input");
    if (residual != nullptr && residual != out && overlap(out, ob, residual, ob))
        return fail(FL_ERR_INVALID_ARG, "out may alias residual only exactly");
    return run_tile(dtype, fl::PRO_ADD, false, A, single_out(W, bias, out, N, (int)act), nullptr, residual, bias_in,
                    nullptr, M, K, 0.f, static_cast<cudaStream_t>(stream));
}

fl_status fl_rms_norm(const void* x, const void* gamma, void* out, int M, int K, float eps, fl_dtype dtype,
                      void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if (!(eps >= 0.0f) || eps > 1e30f) return fail(FL_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (M < 1 || K < 1) return fail(FL_ERR_INVALID_ARG, "fl_rms_norm: sizes must be positive (M=%d K=%d)", M, K);
    if (K % 8 != 0) return fail(FL_ERR_ALIGNMENT, "fl_rms_norm: K must be a multiple of 8 (K=%d)", K);
    fl_status st;
    if ((st = check_ptr("x", x, true)) != FL_OK) return st;
    if ((st = check_ptr("gamma", gamma, true)) != FL_OK) return st;
    if ((st = check_ptr("out", out, true)) != FL_OK) return st;
    const size_t xb = (size_t)M * K * 2;
    if (out != x && overlap(out, xb, x, xb)) return fail(FL_ERR_INVALID_ARG, "out may alias x only exactly");
    if (overlap(out, xb, gamma, (size_t)K * 2)) return fail(FL_ERR_INVALID_ARG, "out overlaps gamma");
    DeviceInfo* di = nullptr;
    if ((st = device_info(&di)) != FL_OK) return st;
    cudaError_t e = fl::launch_rms_norm(dtype, x, gamma, out, M, K, eps, g_opt_pdl.load(), di->sms,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "RMSNorm kernel launch failed: %s", cudaGetErrorString(e));
    count_launch();
    return ok();
}

size_t fl_swiglu_ffn_workspace_size(int M, int F, fl_dtype dtype) {
    (void)dtype;
    if (M < 1 || F < 1) return 0;
    return (size_t)M * (size_t)F * 2;
}

fl_status fl_swiglu_ffn(const void* x, const void* gamma, const void* Wg, const void* Wu, const void* Wd,
                        const void* bias_down, void* out, int M, int D, int F, float eps, void* workspace,
                        size_t workspace_bytes, fl_dtype dtype, void* stream) {
    if (!valid_dtype(dtype)) return fail(FL_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
    if (!(eps >= 0.0f) || eps > 1e30f) return fail(FL_ERR_INVALID_ARG, "eps must be finite and >= 0");
    fl_status st;
    if ((st = check_shape("fl_swiglu_ffn (gate/up)", M, F, D)) != FL_OK) return st;
    if ((st = check_shape("fl_swiglu_ffn (down)", M, D, F)) != FL_OK) return st;
    if ((st = check_ptr("x", x, true)) != FL_OK) return st;
    if ((st = check_ptr("gamma", gamma, true)) != FL_OK) return st;
    if ((st = check_ptr("Wg", Wg, true)) != FL_OK) return st;
    if ((st = check_ptr("Wu", Wu, true)) != FL_OK) return st;
    if ((st = check_ptr("Wd", Wd, true)) != FL_OK) return st;
    if ((st = check_ptr("out", out, true)) != FL_OK) return st;
    if ((st = check_ptr("bias_down", bias_down, false)) != FL_OK) return st;
    if (workspace == nullptr) return fail(FL_ERR_WORKSPACE, "workspace must not be null");
    if (!aligned16(workspace)) return fail(FL_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    const size_t need = fl_swiglu_ffn_workspace_size(M, F, dtype);
    if (workspace_bytes < need)
        return fail(FL_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    const size_t ob = (size_t)M * D * 2, wb = (size_t)F * D * 2;
    const void* ins[6] = {x, gamma, Wg, Wu, Wd, bias_down};
    const size_t insz[6] = {ob, (size_t)D * 2, wb, wb, wb, (size_t)D * 2};
    for (int i = 0; i < 6; ++i) {
        if (overlap(out, ob, ins[i], insz[i])) return fail(FL_ERR_INVALID_ARG, "out overlaps an input");
        if (overlap(workspace, need, ins[i], insz[i])) return fail(FL_ERR_INVALID_ARG, "workspace overlaps an input");
    }
    if (overlap(workspace, need, out, ob)) return fail(FL_ERR_INVALID_ARG, "workspace overlaps out");
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // gate/up: h = silu(RMSNorm(x) Wg^T) * (RMSNorm(x) Wu^T)
    st = run_tile(dtype, fl::PRO_RMS, true, x, single_out(Wg, nullptr, workspace, F, fl::ACT_NONE), Wu, nullptr, gamma,
                  nullptr, M, D, eps, s);
    if (st != FL_OK) return st;
    // down: out = h Wd^T (+ bias_down) + x
    return run_tile(dtype, fl::PRO_NONE, false, workspace, single_out(Wd, bias_down, out, D, fl::ACT_NONE), nullptr, x,
                    nullptr, nullptr, M, F, 0.f, s);
}

fl_status fl_kernel_launches(long long* count) {
    if (count == nullptr) return fail(FL_ERR_INVALID_ARG, "null output pointer");
    *count = g_kernel_launches.load();
    return ok();
}

fl_status fl_launch_cache_stats(long long* hits, long long* misses) {
    if (hits == nullptr || misses == nullptr) return fail(FL_ERR_INVALID_ARG, "null output pointer");
    *hits = g_cache_hits.load();
    *misses = g_cache_misses.load();
    return ok();
}

void fl_launch_cache_clear(void) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    for (CacheSlot& c : g_cache) c.used = false;
}

fl_status fl_device_status(void* stream) {
    DeviceInfo* di = nullptr;
    fl_status st = device_info(&di);
    if (st != FL_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    const size_t off = (size_t)status_slot(di, static_cast<cudaStream_t>(stream)) * sizeof(int);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_fl_status, sizeof(int), off);
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (v == 0) return ok();
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_fl_status, &zero, sizeof(int), off);
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    return fail(FL_ERR_TIMEOUT, "a device-side wait ran past its limit (code %d, wait site %d)", v & 0xff, v >> 8);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// bounded-wait test hook
// ---------------------------------------------------------------------------
namespace {

__global__ void fl_wait_probe_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        uint32_t done;
        // nobody arrives: phase 0 never completes
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a)
            : "memory");
        if (done) return;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > limit_ns) {
            atomicCAS(status, 0, fl::kStatusTimeout | (99 << 8));
            return;
        }
    }
}

}  // namespace

extern "C" fl_status fl_debug_wait_timeout(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(FL_ERR_INVALID_ARG, "limit_us must be 1..1000000");
    DeviceInfo* di = nullptr;
    fl_status st = device_info(&di);
    if (st != FL_OK) return st;
    fl_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        stream_status(di, static_cast<cudaStream_t>(stream)),
                                                                          (unsigned long long)limit_us * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FL_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    count_launch();
    return ok();
}
