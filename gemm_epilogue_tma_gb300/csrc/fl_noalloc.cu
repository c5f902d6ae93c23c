// fl_swiglu_ffn_noalloc: the SwiGLU FFN block for callers that may not
// allocate device memory when they call (an engine that owns a fixed memory
// budget, a plugin whose enqueue must not allocate). The hidden activation h,
// which fl_swiglu_ffn keeps in a caller-provided workspace, lives here in one
// fixed array of this library instead.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdio>
#include <mutex>

#include "../../include/fusedlin.h"
#include "fl_internal.h"

namespace {

// Largest h the array holds: M * F * 2 bytes <= 8 MiB, e.g. 256 tokens at
// F = 11008, or 1024 tokens at F = 4096.
constexpr size_t kScratchBytes = size_t(8) << 20;

// Every GPU that loads the library holds this array until the process exits.
// Host code must not use its name as an address: the name is a host-side
// stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ffn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device (with that device current).
fl_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return (fl_status)fl::set_last_error(FL_ERR_UNSUPPORTED, "fl_swiglu_ffn_noalloc: no CUDA device");
    if (dev < 0 || dev >= kMaxDevices)
        return (fl_status)fl::set_last_error(FL_ERR_UNSUPPORTED, "fl_swiglu_ffn_noalloc: device index out of range");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof(msg), "fl_swiglu_ffn_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return (fl_status)fl::set_last_error(FL_ERR_CUDA, msg);
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return FL_OK;
}

}  // namespace

extern "C" fl_status fl_swiglu_ffn_noalloc(const void* x, const void* gamma, const void* Wg, const void* Wu,
                                           const void* Wd, const void* bias_down, void* out, int M, int D, int F,
                                           float eps, fl_dtype dtype, void* stream) {
    // Host checks that need no device come first, so a rejected call makes no
    // CUDA call at all (fl_swiglu_ffn repeats them with the full set of rules).
    if (dtype != FL_F16 && dtype != FL_BF16)
        return (fl_status)fl::set_last_error(FL_ERR_INVALID_ARG, "fl_swiglu_ffn_noalloc: bad dtype");
    if (M < 1 || D < 1 || F < 1)
        return (fl_status)fl::set_last_error(FL_ERR_INVALID_ARG, "fl_swiglu_ffn_noalloc: sizes must be positive");
    if (x == nullptr || gamma == nullptr || Wg == nullptr || Wu == nullptr || Wd == nullptr || out == nullptr)
        return (fl_status)fl::set_last_error(FL_ERR_INVALID_ARG, "fl_swiglu_ffn_noalloc: a required pointer is null");
    if (fl_swiglu_ffn_workspace_size(M, F, dtype) > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "fl_swiglu_ffn_noalloc: h [%d, %d] needs %zu bytes, more than the library's fixed %zu-byte array; "
                 "use fl_swiglu_ffn with a workspace",
                 M, F, (size_t)M * (size_t)F * 2, kScratchBytes);
        return (fl_status)fl::set_last_error(FL_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    fl_status st = scratch_address(&scratch);
    if (st != FL_OK) return st;
    // h needs no clearing: the gate/up kernel writes every element the down
    // projection reads (the one-launch decode form zeroes its barrier word).
    return fl_swiglu_ffn(x, gamma, Wg, Wu, Wd, bias_down, out, M, D, F, eps, scratch, kScratchBytes, dtype, stream);
}
