// Device helpers shared by the kernels: 16-bit packing, bounded mbarrier
// waits, activations and vector shared-memory access.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fl_internal.h"
#include "fl_ptx.cuh"

namespace fl {

// Phase timestamps for timing studies: compiled in with -DFL_TRACE only;
// slot s of CTA b goes to trace[b * FL_TRACE_SLOTS + s] (16 phase slots; 64
// with -DFL_TRACE_STEPS, whose slots 16-63 time eight K steps of the main
// loop: producer issue, fold hand-off, MMA waits). SM clock cycles, or global
// nanoseconds (comparable across SMs and launches) with -DFL_TRACE_GLOBALTIMER.
#ifdef FL_TRACE
// (read with a memory clobber, so the compiler keeps the mark where it is
// written relative to barriers and memory operations)
__device__ __forceinline__ unsigned long long fl_trace_now() {
    unsigned long long t;
#ifdef FL_TRACE_GLOBALTIMER
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
#else
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t)::"memory");
#endif
    return t;
}
#define FL_TRACE_NOW() fl_trace_now()
#ifdef FL_TRACE_STEPS
#define FL_TRACE_SLOTS 64
#else
#define FL_TRACE_SLOTS 16
#endif
#define FL_MARK(p, slot)                                                                   \
    do {                                                                                   \
        if ((p).trace != nullptr)                                                          \
            (p).trace[blockIdx.x * FL_TRACE_SLOTS + (slot)] = (unsigned long long)FL_TRACE_NOW(); \
    } while (0)
#else
#define FL_MARK(p, slot) \
    do {                 \
    } while (0)
#endif
// Per-step marks: K step j (8 <= j < 16 of a CTA's first tile) into slot base + j - 8.
#ifdef FL_TRACE_STEPS
#define FL_MARK_STEP(p, base, j)                                  \
    do {                                                          \
        if ((j) >= 8 && (j) < 16) FL_MARK(p, (base) + (j) - 8);   \
    } while (0)
#else
#define FL_MARK_STEP(p, base, j) \
    do {                         \
    } while (0)
#endif

template <int DT>
struct DTypeOps;

template <>
struct DTypeOps<DT_F16> {
    static constexpr uint32_t kFormat = 0;
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        return __half22float2(*reinterpret_cast<__half2*>(&u));
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
    // a + b per 16-bit lane, rounded once (IEEE addition)
    __device__ static __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        __half2 r = __hadd2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
};

template <>
struct DTypeOps<DT_BF16> {
    static constexpr uint32_t kFormat = 1;
    __device__ static __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    // Widening as the mixed-precision FMA x * 1 + (-0) (fp32 result, bf16
    // factors; sm_100 and later), which is exact. In the LayerNorm fold it
    // measured 4 % faster than shifting the halves into place, which in turn
    // beat the library conversion.
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        float2 r;
        asm("{\n\t.reg .b16 lo, hi, one;\n\tmov.b32 {lo, hi}, %2;\n\tmov.b16 one, 0x3F80;\n\t"
            "fma.rn.f32.bf16 %0, lo, one, 0f80000000;\n\tfma.rn.f32.bf16 %1, hi, one, 0f80000000;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(u));
        return r;
    }
    __device__ static __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
    __device__ static __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hadd2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// Waits for the phase of parity `parity` of `bar`. Gives up (returns false)
// after timeout_ns, or early once another role has recorded a failure.
static __device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, int* status,
                                           unsigned long long timeout_ns, int where) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*reinterpret_cast<volatile int*>(status) != 0) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                atomicCAS(status, 0, kStatusTimeout | (where << 8));
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* status,
                                         unsigned long long timeout_ns, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, status, timeout_ns, where);
}

// Bounded wait with cluster-scope acquire, for barriers a peer CTA arrives on.
static __device__ __noinline__ bool wait_bar_cluster_slow(uint32_t bar, uint32_t parity, int* status,
                                                          unsigned long long timeout_ns, int where) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 1023) == 0) {
            if (*reinterpret_cast<volatile int*>(status) != 0) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                atomicCAS(status, 0, kStatusTimeout | (where << 8));
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, int* status,
                                                 unsigned long long timeout_ns, int where) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return wait_bar_cluster_slow(bar, parity, status, timeout_ns, where);
}

// Time-bounded only: used while draining after a failure.
static __device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, unsigned long long ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > ns) return false;
    }
    return true;
}

// Output of a global column block: the outputs of a launch lie side by side
// along N, output i taking column blocks [nb0[i], nb0[i + 1]).
struct OutSel {
    int oi;  // output index
    int nb;  // column block within that output
};

__device__ __forceinline__ OutSel out_sel(const GemmParams&, int nb) { return OutSel{0, nb}; }

__device__ __forceinline__ OutSel out_sel(const GemmParamsMulti& p, int nb) {
    int oi = 0;
#pragma unroll
    for (int i = 1; i < kMaxOut; ++i)
        if (i < p.n_out && nb >= p.nb0[i]) oi = i;
    return OutSel{oi, nb - p.nb0[oi]};
}

// Fields of output oi: a single-output launch has only output 0.
__device__ __forceinline__ const CUtensorMap* tm_b(const GemmParams& p, int) { return &p.tmB; }
__device__ __forceinline__ const CUtensorMap* tm_out(const GemmParams& p, int) { return &p.tmOut; }
__device__ __forceinline__ const void* out_bias(const GemmParams& p, int) { return p.bias; }
__device__ __forceinline__ void* out_ptr(const GemmParams& p, int) { return p.out_ptr; }
__device__ __forceinline__ int out_n(const GemmParams& p, int) { return p.N; }
__device__ __forceinline__ int out_act(const GemmParams& p, int) { return p.act; }
__device__ __forceinline__ const CUtensorMap* tm_b(const GemmParamsMulti& p, int oi) {
    return oi == 0 ? &p.tmB : &p.tmBx[oi - 1];
}
__device__ __forceinline__ const CUtensorMap* tm_out(const GemmParamsMulti& p, int oi) {
    return oi == 0 ? &p.tmOut : &p.tmOutx[oi - 1];
}
__device__ __forceinline__ const void* out_bias(const GemmParamsMulti& p, int oi) {
    return oi == 0 ? p.bias : p.biasx[oi - 1];
}
__device__ __forceinline__ void* out_ptr(const GemmParamsMulti& p, int oi) {
    return oi == 0 ? p.out_ptr : p.out_ptrx[oi - 1];
}
__device__ __forceinline__ int out_n(const GemmParamsMulti& p, int oi) { return oi == 0 ? p.N : p.Nx[oi - 1]; }
__device__ __forceinline__ int out_act(const GemmParamsMulti& p, int oi) { return oi == 0 ? p.act : p.actx[oi - 1]; }

// Hardware tanh (one special-function op; relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GeLU (tanh form) and SiLU both as h (1 + tanh(u)) with h = v / 2:
//   GeLU: u = sqrt(2/pi) (v + 0.044715 v^3);  SiLU: v sigmoid(v), u = v / 2.
// One special-function op per element (the epilogue of a 128 x 256 tile
// issues 32 K of them, at 16 per SM cycle).
__device__ __forceinline__ float act_apply(int act, float v) {
    switch (act) {
        case ACT_GELU: {
            const float k = 0.7978845608028654f;  // sqrt(2 / pi)
            const float h = 0.5f * v;
            return fmaf(h, tanh_approx(k * fmaf(0.044715f * v, v * v, v)), h);
        }
        case ACT_SILU: {
            const float h = 0.5f * v;
            return fmaf(h, tanh_approx(h), h);
        }
        case ACT_RELU:
            return fmaxf(v, 0.0f);
        default:
            return v;
    }
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

}  // namespace fl
