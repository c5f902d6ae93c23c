/*
 * libfusedlin: fused transformer dense layer on GB300 (sm_103a).
 *
 * One GEMM with FP32 accumulation on fp16/bf16 operands, with an optional
 * RMSNorm / LayerNorm prologue on the activation rows and a bias /
 * activation / residual / SwiGLU epilogue, all applied on-chip: the
 * normalised activation and the pre-activation never pass through device
 * memory.
 *
 * Operations (sources, by page and section):
 *   - The nine fused patterns of the llm-fusion-compiler README, pattern
 *     table "Pattern / Operations fused": gemm_bias_gelu, gemm_bias_silu,
 *     gemm_bias_relu, gemm_bias, gemm_bias_residual, gemm_gelu, gemm_silu,
 *     layernorm_gemm, rmsnorm_gemm. GeLU is the tanh ("fast approximation")
 *     form: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))).
 *   - RMSNorm feeding a linear projection: the LLMBoost README, op
 *     llm.fused_rmsnorm_linear(x, w_norm, w_proj, epsilon) (section 1) and
 *     its CUDA kernel, 1/rms = rsqrt(sum(x^2)/d_in + epsilon) (section 3);
 *     the same eps-inside-the-root form as the RMSNorm loop nest of the
 *     "hackable compiler" post.
 *   - The SwiGLU FFN block of the llm-fusion-compiler README ("FFN block
 *     (SwiGLU style)": three GEMMs, activation, elementwise product, bias,
 *     residual) in its Llama form: RMSNorm, gate and up projections,
 *     silu(gate) * up, down projection, plus the pre-norm input.
 *
 * Conventions for every entry point:
 *   - Layouts are row-major and dense: A/x [M, K]; weights W [N, K] (the
 *     linear-layer layout: out = act(A W^T + bias) ...); bias [N];
 *     residual and out [M, N]; gamma, beta [K].
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned. K and N (and D, F for the FFN) must be multiples of 8 so that
 *     every row starts on a 16-byte boundary. M may be any value >= 1.
 *   - dtype selects fp16 or bf16 for every tensor of the call; accumulation
 *     and the epilogue arithmetic are fp32; the output is rounded to nearest
 *     even.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Every call is asynchronous on that stream.
 *   - Device memory: fl_gemm_epilogue and the RMS form of fl_norm_gemm allocate
 *     nothing. The LayerNorm form of fl_norm_gemm takes 8 bytes per row of
 *     stream-ordered scratch for its row statistics from a library-owned
 *     memory pool and frees it on the stream after the GEMM (see there).
 *     fl_swiglu_ffn keeps its hidden activation in a caller-provided
 *     workspace; fl_swiglu_ffn_noalloc keeps it in a fixed 8 MiB array of the
 *     library instead. The library's other device state is a small table
 *     of status words (one per stream, see fl_device_status).
 *   - out may alias residual exactly (same pointer); no other aliasing of an
 *     output with an input is allowed.
 *   - Errors: a call that fails validation returns a non-zero fl_status
 *     before launching anything and writes nothing; fl_last_error() then
 *     returns a message (per thread). A device-side wait that exceeds its time
 *     limit makes the kernel stop early and record FL_ERR_TIMEOUT in the
 *     status word of its stream, which fl_device_status() reads (see there).
 */
#ifndef FUSEDLIN_H
#define FUSEDLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FL_OK = 0,
    FL_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad enum, forbidden aliasing */
    FL_ERR_UNSUPPORTED = 2, /* no sm_103a device, or a size beyond what the kernels handle */
    FL_ERR_ALIGNMENT = 3,   /* pointer not 16-byte aligned, or K/N/D/F not a multiple of 8 */
    FL_ERR_WORKSPACE = 4,   /* FFN workspace missing or smaller than fl_swiglu_ffn_workspace_size */
    FL_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed (message in fl_last_error) */
    FL_ERR_TIMEOUT = 6      /* a device-side wait ran past its limit (from fl_device_status) */
} fl_status;

typedef enum { FL_F16 = 0, FL_BF16 = 1 } fl_dtype;

/* The nine fused patterns, in the order of the llm-fusion-compiler pattern table. */
typedef enum {
    FL_GEMM_BIAS_GELU = 0,     /* gelu_tanh(A W^T + bias)          */
    FL_GEMM_BIAS_SILU = 1,     /* silu(A W^T + bias)               */
    FL_GEMM_BIAS_RELU = 2,     /* relu(A W^T + bias)               */
    FL_GEMM_BIAS = 3,          /* A W^T + bias                     */
    FL_GEMM_BIAS_RESIDUAL = 4, /* A W^T + bias + residual          */
    FL_GEMM_GELU = 5,          /* gelu_tanh(A W^T)                 */
    FL_GEMM_SILU = 6,          /* silu(A W^T)                      */
    FL_LAYERNORM_GEMM = 7,     /* LayerNorm(A) W^T  (fl_norm_gemm) */
    FL_RMSNORM_GEMM = 8        /* RMSNorm(A) W^T    (fl_norm_gemm) */
} fl_pattern;

typedef enum { FL_NORM_RMS = 0, FL_NORM_LAYER = 1 } fl_norm_kind;

typedef enum { FL_ACT_NONE = 0, FL_ACT_GELU_TANH = 1, FL_ACT_SILU = 2, FL_ACT_RELU = 3 } fl_act;

/*
 * out[M,N] = epilogue(A[M,K] W[N,K]^T) for the seven GEMM-first patterns
 * (FL_GEMM_BIAS_GELU .. FL_GEMM_SILU); llm-fusion-compiler pattern table.
 *   bias:     [N], required by the *_BIAS* patterns, ignored otherwise.
 *   residual: [M,N], required by FL_GEMM_BIAS_RESIDUAL, ignored otherwise;
 *             may be the same pointer as out.
 * Epilogue order: accumulate, + bias, activation, + residual, round.
 * FL_LAYERNORM_GEMM / FL_RMSNORM_GEMM return FL_ERR_INVALID_ARG here: they
 * need gamma/beta/eps and are served by fl_norm_gemm.
 */
fl_status fl_gemm_epilogue(const void* A, const void* W, const void* bias, const void* residual,
                           void* out, int M, int N, int K, fl_pattern pattern, fl_dtype dtype,
                           void* stream);

/*
 * out[M,N] = act(norm(x)[M,K] W[N,K]^T + bias) with the norm as prologue;
 * the rmsnorm_gemm / layernorm_gemm patterns of the llm-fusion-compiler
 * table, generalised with an optional bias and activation.
 *   FL_NORM_RMS:   norm(x) = x * gamma / sqrt(mean_k(x^2) + eps)
 *                  (LLMBoost CUDA kernel section: rsqrt(ss / d_in + eps)).
 *   FL_NORM_LAYER: norm(x) = (x - mean) / sqrt(var + eps) * gamma + beta,
 *                  biased variance.
 *   gamma: [K], required. beta: [K], LayerNorm only, NULL means zero;
 *   ignored for RMS. bias: [N] or NULL. eps must be finite and >= 0.
 * The RMS statistics are computed from the fp16/bf16 input in fp32; gamma is
 * folded into the staged operand (one rounding to the dtype) and 1/rms is
 * applied to the fp32 accumulator as a row scale.
 * LayerNorm first runs a small statistics kernel on `stream` that writes each
 * row's mean and 1/sqrt(var + eps) (fp32, shifted sums) to M * 8 bytes of
 * scratch taken from a library-owned stream-ordered memory pool and freed on
 * `stream` after the GEMM kernel; the GEMM kernel then folds
 * (x - mean) * rstd * gamma + beta into its staged operand (one rounding).
 * Works under CUDA graph capture; returns FL_ERR_CUDA if the scratch cannot
 * be allocated.
 */
fl_status fl_norm_gemm(const void* x, const void* gamma, const void* beta, const void* W,
                       const void* bias, void* out, int M, int N, int K, float eps,
                       fl_norm_kind norm_kind, fl_act act, fl_dtype dtype, void* stream);

/* Most outputs one fl_norm_gemm_multi call computes. */
#define FL_MAX_OUTPUTS 4

/*
 * Several consumers of one normalised activation in one launch (horizontal
 * fusion: operators sharing a common input, the inferensys "Fusion Compiler"
 * glossary, fusion groups). For i < n_out:
 *   out_i[M, N_i] = act_i(norm(x)[M, K] W_i[N_i, K]^T + bias_i)
 * with norm(x) as in fl_norm_gemm. This is the case the LLMBoost README's
 * "one-user safety guard" leaves unfused (a normalised tensor with two or
 * more consumers, e.g. the Q, K and V projections or an MoE gate): here the
 * LayerNorm statistics are computed once for all outputs, the RMS statistics
 * come with the fold, and every output's tiles share one launch (one grid
 * over the outputs side by side along N), so no consumer waits for another
 * and none rereads a materialised norm(x).
 *   n_out:  1 .. FL_MAX_OUTPUTS.
 *   W[i]:   [N_i, K] device pointers; out[i]: [M, N_i] device pointers.
 *   bias:   NULL (no bias anywhere) or an array whose entries are [N_i] or NULL.
 *   N[i]:   multiples of 8. act: NULL (no activation) or one fl_act per output.
 * The arrays themselves are host memory, read during the call only. Outputs
 * may not overlap each other or any input. Memory and errors as fl_norm_gemm.
 */
fl_status fl_norm_gemm_multi(const void* x, const void* gamma, const void* beta, int n_out,
                             const void* const* W, const void* const* bias, void* const* out,
                             const int* N, const int* act, int M, int K, float eps,
                             fl_norm_kind norm_kind, fl_dtype dtype, void* stream);

/*
 * Elementwise input prologue (the "hackable compiler" post's example
 * torch.relu(torch.matmul(x + bias, w)), whose prologue adds a bias along K
 * inside the reduction loop):
 *   out[M,N] = act((A[M,K] + bias_in[K]) W[N,K]^T + bias[N]) (+ residual[M,N])
 * A + bias_in is formed in the staged operand (rounded once to the dtype) and
 * never stored. bias_in: required. bias, residual: [N], [M,N] or NULL;
 * residual may be the same pointer as out. Epilogue order as fl_gemm_epilogue.
 * Allocates nothing.
 */
fl_status fl_input_bias_gemm(const void* A, const void* bias_in, const void* W, const void* bias,
                             const void* residual, void* out, int M, int N, int K, fl_act act,
                             fl_dtype dtype, void* stream);

/*
 * Standalone RMSNorm, out[M,K] = x * gamma / sqrt(mean_k(x^2) + eps), computed
 * in fp32 and rounded once: the generated RMSNorm kernel of the "hackable
 * compiler" post (sum of squares, times 1/K, plus eps, rsqrt, times x, times
 * the weight). For a normalised tensor with more consumers than
 * fl_norm_gemm_multi takes, or consumers that are not GEMMs. out may be x
 * itself (in place) but may not otherwise overlap x or gamma. K must be a
 * multiple of 8. Allocates nothing. Bound by HBM bandwidth.
 */
fl_status fl_rms_norm(const void* x, const void* gamma, void* out, int M, int K, float eps,
                      fl_dtype dtype, void* stream);

/* Bytes of workspace fl_swiglu_ffn needs: the hidden activation h [M,F] in the
 * dtype, M * F * 2 (0 when M or F is below 1). */
size_t fl_swiglu_ffn_workspace_size(int M, int F, fl_dtype dtype);

/*
 * Llama-style SwiGLU FFN block (llm-fusion-compiler "FFN block (SwiGLU
 * style)"):
 *   xh  = RMSNorm(x; gamma, eps)                 x [M,D], gamma [D]
 *   h   = silu(xh Wg^T) * (xh Wu^T)              Wg, Wu [F,D]; h [M,F] in dtype
 *   out = h Wd^T (+ bias_down) + x               Wd [D,F], bias_down [D] or NULL
 * Two launches: a gate/up kernel that feeds one staged activation tile to both
 * weights and writes h, then a down-projection kernel with a residual
 * epilogue (for 1 to 8 rows both on the decode kernel, where its activation
 * rows fit in shared memory; see FL_OPT_VARIANT). workspace: device memory of at least
 * fl_swiglu_ffn_workspace_size(M, F, dtype) bytes, 16-byte aligned, owned by
 * the caller; its contents on return are h. out must not alias x.
 */
fl_status fl_swiglu_ffn(const void* x, const void* gamma, const void* Wg, const void* Wu,
                        const void* Wd, const void* bias_down, void* out, int M, int D, int F,
                        float eps, void* workspace, size_t workspace_bytes, fl_dtype dtype,
                        void* stream);

/*
 * fl_swiglu_ffn without a workspace argument, for callers that may not
 * allocate device memory at call time: an inference engine or plugin that
 * owns a fixed, pre-planned memory budget, or code that runs where an
 * allocation is not allowed. The pages have no counterpart; this is a
 * library convenience.
 *   Arguments and results are those of fl_swiglu_ffn; the hidden activation
 *   h [M,F] is kept in one fixed 8 MiB device array that the library holds on
 *   every GPU that loads it, until the process exits. M * F * 2 must be at
 *   most 8 MiB (for example M = 256 at F = 11008); larger calls return
 *   FL_ERR_WORKSPACE without launching.
 *   The call allocates nothing. Its first call on a device looks up the
 *   array's device address for that device (cudaGetSymbolAddress); under
 *   lazy module loading that lookup is also what loads the library's device
 *   code and reserves the 8 MiB. So make the first call on each device at
 *   initialisation time, before any stream capture. Sizes, dtype and
 *   pointers are checked on the host before that lookup: a rejected call
 *   makes no CUDA call.
 *   All calls share the array and it keeps the last call's h: two calls whose
 *   kernels overlap on the GPU (different streams, or different host threads)
 *   race on it and give wrong results.
 */
fl_status fl_swiglu_ffn_noalloc(const void* x, const void* gamma, const void* Wg, const void* Wu,
                                const void* Wd, const void* bias_down, void* out, int M, int D,
                                int F, float eps, fl_dtype dtype, void* stream);

/*
 * The dense part of a Llama-style decoder layer as a prepared call sequence.
 * At decode sizes every kernel of a layer takes a few microseconds, so host
 * launch costs weigh as much as the kernels; a decode step is meant to be
 * captured once, every layer with the caller's attention in between, into
 * one CUDA graph (fl_capture_begin .. fl_capture_end) and replayed with one
 * launch (the "Fusion Compiler" glossary pairs fusion with CUDA Graph capture
 * as the coarse-grained launch optimisation). The layer is split where the
 * attention core sits, which this library does not compute:
 *   half 0:  q, k, v = RMSNorm(x; gamma_attn) [Wq; Wk; Wv]^T       (fl_norm_gemm_multi)
 *   ... the caller's attention reads q, k, v and writes attn ...
 *   half 1:  h   = attn Wo^T (+ bias_o) + x                        (fl_gemm_epilogue)
 *            out = silu(hn Wg^T) * (hn Wu^T) Wd^T + h, hn = RMSNorm(h; gamma_ffn)   (fl_swiglu_ffn)
 * Shapes: x, attn, h, out, q [M, D]; k, v [M, Dkv]; Wq, Wo [D, D];
 * Wk, Wv [Dkv, D]; Wg, Wu [F, D]; Wd [D, F]; gamma_* and bias_o [D]. All are
 * caller-owned device pointers, fixed for the life of the layer. bias_o may
 * be NULL (no bias). eps is the RMSNorm epsilon of both norms.
 */
typedef struct {
    fl_dtype dtype;
    int M, D, Dkv, F;
    float eps;
    const void* x;
    const void* gamma_attn;
    const void* Wq;
    const void* Wk;
    const void* Wv;
    void* q;
    void* k;
    void* v;
    const void* attn;
    const void* Wo;
    const void* bias_o;
    void* h;
    const void* gamma_ffn;
    const void* Wg;
    const void* Wu;
    const void* Wd;
    void* out;
} fl_layer_desc;

typedef struct fl_layer fl_layer;

/*
 * Validates the description, allocates the layer's own device memory (the
 * FFN hidden activation, M * F * 2 bytes, and D zeros when bias_o is NULL)
 * and runs both halves once on an internal stream (the one-time kernel
 * set-up; this writes q, k, v, h and out from whatever x and attn hold), so
 * that every later call of the layer hits the launch cache. Call it at
 * initialisation, not inside a stream capture. On failure *layer is NULL and
 * nothing is left allocated.
 */
fl_status fl_layer_create(const fl_layer_desc* desc, fl_layer** layer);

/* Issues half 0 or 1 on `stream` (capturable); allocates nothing. */
fl_status fl_layer_issue(const fl_layer* layer, int half, void* stream);

/* Frees the layer's device memory and stream. NULL is a no-op. */
void fl_layer_destroy(fl_layer* layer);

/*
 * Capture of library calls (and any other work the caller issues on the same
 * stream from the same thread) into one CUDA graph: fl_capture_begin starts
 * a thread-local capture of `stream`; fl_capture_end ends it, instantiates
 * and uploads the graph and returns its handle (*graph_exec, a
 * cudaGraphExec_t); fl_graph_launch replays it on a stream; fl_graph_destroy
 * frees it (NULL is a no-op). Every call of this library except
 * fl_layer_create and fl_device_status may be captured; the first call of a
 * kernel configuration should come before the capture (its one-time set-up
 * is not capturable), which fl_layer_create does for a layer.
 */
fl_status fl_capture_begin(void* stream);
fl_status fl_capture_end(void* stream, void** graph_exec);
fl_status fl_graph_launch(void* graph_exec, void* stream);
void fl_graph_destroy(void* graph_exec);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* fl_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the status word of `stream`,
 * which this library's kernels launched on that stream set when a bounded
 * wait runs out. Returns FL_OK, FL_ERR_TIMEOUT, or FL_ERR_CUDA if the
 * synchronisation itself failed.
 * Each device keeps 64 status words: word 0 for the legacy default stream
 * (NULL), then one per stream handle in the order the library first sees
 * them; the 64th distinct handle and later ones share word 0. A kernel
 * captured into a graph keeps the word of the stream it was captured on,
 * wherever the graph is replayed. The word is sticky: until it is read, a
 * later kernel on the same stream whose wait is slow gives up at once.
 */
fl_status fl_device_status(void* stream);

/*
 * Tuning overrides, for benchmarks and tests. They are process-wide: each value
 * is stored and read atomically, and a change applies to the calls any thread
 * prepares after it (a call repeated from the launch cache keeps the choice
 * it was prepared with only while the options are unchanged: they are part
 * of the cache key).
 *   FL_OPT_TILE_N:      0 = automatic, else the CTA tile width (128 or 256).
 *   FL_OPT_VARIANT:     0 = automatic, 1 = tile kernel, 2 = small-M split-K kernel
 *                       (for the SwiGLU gate/up GEMM only up to 64 rows, else
 *                       the tile kernel), 3 = CTA-pair kernel (256 x 256 tiles
 *                       on two SMs; for the gate/up kernel, Wg and Wu rows
 *                       stacked in one tile), 4 = the decode kernel (1 to 8
 *                       rows; weight-streaming warp-level MMAs; the
 *                       transformed activation rows must fit in 96 KB of
 *                       shared memory). Automatic choice
 *                       takes the decode kernel where it fits for 1 to 4
 *                       rows, and for 5 to 8 rows when K <= 2048 or the
 *                       call is neither LayerNorm nor the SwiGLU gate/up
 *                       pair.
 *   FL_OPT_TIMEOUT_MS:  limit of every device-side wait (default 2000).
 *   FL_OPT_SPLIT_K:     0 = automatic, else the K split of the small-M kernel (1..8).
 *   FL_OPT_PDL:         1 (default) = launch each kernel with a programmatic
 *                       dependency on the previous kernel of the stream, so its
 *                       set-up overlaps that kernel's tail (all of its memory
 *                       accesses still wait for it); 0 = plain stream order.
 *   FL_OPT_LAUNCH_CACHE: 1 (default) = keep the prepared launch (kernel choice
 *                       and encoded tensor maps) of each recent argument set,
 *                       so a call repeated with the same pointers, sizes and
 *                       options skips that host work (see fl_launch_cache_stats);
 *                       0 = prepare every call afresh.
 *   FL_OPT_WEIGHT_PRELOAD: 0 (default) or 1. With 1 the caller promises that
 *                       no kernel on the stream writes the weight matrix W
 *                       between its last host-ordered write and this call (the
 *                       usual case: weights are read-only across a layer
 *                       sequence). The small-M split-K kernel then stages its
 *                       first weight tiles into shared memory before its
 *                       programmatic dependency on the previous kernel
 *                       resolves, so the weight stream of a decode step starts
 *                       while the previous layer finishes (the other kernels,
 *                       which hold their SMs to the end of a grid, gained
 *                       nothing from it). Activations, gamma, beta, bias and
 *                       residual are still read only after it.
 * Returns FL_ERR_INVALID_ARG for an unknown key or a value out of range.
 */
typedef enum {
    FL_OPT_TILE_N = 0,
    FL_OPT_VARIANT = 1,
    FL_OPT_TIMEOUT_MS = 2,
    FL_OPT_SPLIT_K = 3,
    FL_OPT_PDL = 4,
    FL_OPT_WEIGHT_PRELOAD = 5,
    FL_OPT_LAUNCH_CACHE = 6
} fl_option;
fl_status fl_set_option(fl_option key, int value);

/*
 * Host-side launch cache. Every fused call first validates its arguments,
 * then needs a kernel choice and the TMA tensor maps of its operands (a
 * driver call per map). Both depend only on the call's pointers, sizes, dtype
 * and options, so the library keeps them for the last 64 argument sets (one
 * slot per set, replaced on collision) and a repeated call only looks them up
 * and launches; the mutable per-call state (the LayerNorm scratch) is set at
 * launch. fl_launch_cache_stats returns the hits and misses since the library
 * was loaded; fl_launch_cache_clear forgets every entry (e.g. after freeing
 * buffers whose addresses may be reused with other contents: entries hold
 * addresses and shapes only, never data, so a stale entry is still correct
 * for the same address and shape).
 */
fl_status fl_launch_cache_stats(long long* hits, long long* misses);
void fl_launch_cache_clear(void);

/*
 * Kernels this library has launched since it was loaded (every thread and
 * device together): incremented on the host after each successful kernel
 * launch call, including launches recorded into a stream capture (a replayed
 * graph adds nothing). *count = the total; FL_ERR_INVALID_ARG if count is
 * NULL.
 */
fl_status fl_kernel_launches(long long* count);

/*
 * Test hook for the bounded-wait machinery: launches one CTA that waits on a
 * device barrier that nothing ever completes, with a limit of `limit_us`
 * microseconds (1..1000000). The kernel gives up, records FL_ERR_TIMEOUT in the
 * status word of `stream` and returns; the GPU context stays usable. Follow it
 * with fl_device_status(stream) to read (and clear) the status.
 */
fl_status fl_debug_wait_timeout(int limit_us, void* stream);

/* Library version string. */
const char* fl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSEDLIN_H */
