// Shared device/host helpers of the MoE library (element types, vector IO, error word,
// bounded waits, launch accounting). Nothing here knows about the layer's arithmetic.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <algorithm>
#include <atomic>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- device error word
enum : int { kErrNone = 0, kErrTimeout = 1, kErrBounds = 2 };

__device__ __forceinline__ void raise_error(int* err, int code) {
    if (err) atomicCAS(err, kErrNone, code);
}

// Cycle budget of every spin-wait (~2 s at 2 GHz): a wait that runs out records
// kErrTimeout and returns false so the kernel can unwind instead of hanging.
constexpr long long kSpinBudgetCycles = 4000000000LL;

// ---------------------------------------------------------------- dependent launches
// Kernels are launched with programmatic stream serialization: a kernel may start (and run
// its prologue) while the previous kernel of its stream finishes. Every kernel therefore
// calls pdl_wait() before its first access to global memory that another kernel writes or
// reads; the wait returns once the previous kernel has completed and its writes are visible
// (immediately when there is none). It then lets the next kernel of the stream launch.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- kernel trace (host)
// While the calling host thread has a trace open (moe_trace_begin), each kernel launch on a
// stream that is not being captured is bracketed by two timing events on its stream, so that
// moe_trace_end can report every kernel's own device time. Off otherwise: one thread-local
// test per launch.
extern thread_local bool t_trace_on;
int trace_before(const void* fn, cudaStream_t s);    // record slot, or -1
void trace_after(int slot, cudaStream_t s);

// cudaLaunchKernelEx with the trace hooks around it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(const cudaLaunchConfig_t& cfg, void (*kern)(KArgs...), Args... args) {
    const int slot = t_trace_on ? trace_before(reinterpret_cast<const void*>(kern), cfg.stream) : -1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (slot >= 0) trace_after(slot, cfg.stream);
    return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return launch_ex(cfg, kern, args...);
}

// p[0..n) = v as a kernel, so that it orders with the dependent launches around it like any
// other kernel of the stream.
template <typename V>
__global__ void __launch_bounds__(256) fill_kernel(V* __restrict__ p, long long n, V v) {
    pdl_wait();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        p[i] = v;
}

// ---------------------------------------------------------------- element types
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <typename T> __device__ __forceinline__ float ld_f(const T* p) { return Elem<T>::to_f(*p); }
template <typename T> __device__ __forceinline__ void st_f(T* p, float v) { *p = Elem<T>::from_f(v); }

// 16-byte vector of elements: 8 bf16 or 4 fp32.
template <typename T> struct Vec16 { static constexpr int N = 16 / sizeof(T); };

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* out) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    } else {
        out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
        out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
    }
}

// The 16 bytes of a load16, already fetched.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* out) {
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    } else {
        out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
        out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
    }
}

template <typename T>
__device__ __forceinline__ void store16(T* p, const float* in) {
    uint4 u;
    if constexpr (sizeof(T) == 2) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
    } else {
        u.x = __float_as_uint(in[0]); u.y = __float_as_uint(in[1]);
        u.z = __float_as_uint(in[2]); u.w = __float_as_uint(in[3]);
    }
    *reinterpret_cast<uint4*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// GELU(a) = a * Phi(a) with the exact erf form and its derivative Phi(a) + a * phi(a), both
// from one exponential. erf(x) for x >= 0 uses the rational-times-exponential form of
// Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.26:
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),  t = 1 / (1 + p x),
// absolute error <= 1.5e-7; with x = |a| / sqrt(2), exp(-x^2) = exp(-a^2 / 2) = sqrt(2 pi) phi(a).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void gelu_and_grad_f(float a, float& g, float& gp) {
    // hardware reciprocal and base-2 exponential (relative error ~2^-22): far below the
    // formula's 1.5e-7. The 1/2 of Phi = (1 + erf) / 2 is folded into the coefficients:
    // h = 0.5 (a1 t + ... + a5 t^5) exp(-a^2/2) = 0.5 erfc(|a| / sqrt 2).
    const float t = rcp_approx(fmaf(0.3275911f * 0.70710678118654752f, fabsf(a), 1.0f));
    float q = fmaf(0.5f * 1.061405429f, t, 0.5f * -1.453152027f);
    q = fmaf(q, t, 0.5f * 1.421413741f);
    q = fmaf(q, t, 0.5f * -0.284496736f);
    q = fmaf(q, t, 0.5f * 0.254829592f);
    const float e = ex2_approx(a * a * -0.72134752044448170f);   // exp(-a^2/2) = 2^(-a^2 log2(e) / 2)
    const float h = (q * t) * e;
    const float Phi = a >= 0.f ? 1.0f - h : h;                     // standard normal CDF
    g = a * Phi;
    gp = fmaf(a * 0.39894228040143268f, e, Phi);                  // Phi + a phi(a)
}

// ---- packed fp32 pairs: Blackwell's f32x2 add/mul/fma issue two IEEE fp32 operations (round
// to nearest, no flush) per instruction. A pair lives in one 64-bit register pair.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t splat2(float c) { return pk2(c, c); }

// gelu_and_grad_f on two values at once: the same formula and constants, with the
// polynomial, the products and the final combination in f32x2 operations (the reciprocal and
// the exponential stay per element on the special-function unit).
__device__ __forceinline__ void gelu_and_grad_f2(float a0, float a1, float& g0, float& g1, float& gp0,
                                                 float& gp1) {
    const uint64_t a = pk2(a0, a1);
    const float p = 0.3275911f * 0.70710678118654752f;
    const uint64_t t = pk2(rcp_approx(fmaf(p, fabsf(a0), 1.0f)), rcp_approx(fmaf(p, fabsf(a1), 1.0f)));
    uint64_t q = fma2(splat2(0.5f * 1.061405429f), t, splat2(0.5f * -1.453152027f));
    q = fma2(q, t, splat2(0.5f * 1.421413741f));
    q = fma2(q, t, splat2(0.5f * -0.284496736f));
    q = fma2(q, t, splat2(0.5f * 0.254829592f));
    float r0, r1;
    upk2(mul2(mul2(a, a), splat2(-0.72134752044448170f)), r0, r1);   // -a^2 log2(e) / 2
    const uint64_t e = pk2(ex2_approx(r0), ex2_approx(r1));           // exp(-a^2/2)
    const uint64_t h = mul2(mul2(q, t), e);                            // 0.5 erfc(|a| / sqrt 2)
    float h0, h1, o0, o1;
    upk2(h, h0, h1);
    upk2(fma2(h, splat2(-1.0f), splat2(1.0f)), o0, o1);               // 1 - h
    const uint64_t Phi = pk2(a0 >= 0.f ? o0 : h0, a1 >= 0.f ? o1 : h1);
    upk2(mul2(a, Phi), g0, g1);
    upk2(fma2(mul2(a, splat2(0.39894228040143268f)), e, Phi), gp0, gp1);
}

__device__ __forceinline__ float gelu_f(float a) {
    return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_grad_f(float a) {
    const float Phi = 0.5f * (1.0f + erff(a * 0.70710678118654752f));
    const float phi = 0.39894228040143268f * __expf(-0.5f * a * a);
    return Phi + a * phi;
}

// Training-time routing noise: a standard normal per (token, expert), four experts per draw of
// the Philox4x64-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011). Experts 4g .. 4g + 3 of token t take counter
// (t, g, 0, 0) with key (seed, 0); the top 24 bits of outputs 0, 1 and of outputs 2, 3 give two
// (u1, u2) pairs in (0, 1], and Box-Muller turns each pair into the two normals
// sqrt(-2 ln u1) cos(2 pi u2) and sqrt(-2 ln u1) sin(2 pi u2), in that order.
__device__ __forceinline__ void routing_noise4(int t, int g, uint32_t seed, float (&z)[4]) {
    uint64_t c0 = (uint64_t)(uint32_t)t, c1 = (uint64_t)(uint32_t)g, c2 = 0, c3 = 0;
    uint64_t k0 = seed, k1 = 0;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t lo0 = 0xD2E7470EE14C6C93ull * c0, hi0 = __umul64hi(0xD2E7470EE14C6C93ull, c0);
        const uint64_t lo1 = 0xCA5A826395121157ull * c2, hi1 = __umul64hi(0xCA5A826395121157ull, c2);
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    const uint64_t o[4] = {c0, c1, c2, c3};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float u1 = (float)((uint32_t)(o[2 * h] >> 40) + 1u) * 5.9604644775390625e-8f;   // 2^-24
        const float u2 = (float)((uint32_t)(o[2 * h + 1] >> 40) + 1u) * 5.9604644775390625e-8f;
        const float r = sqrtf(-2.0f * logf(u1));
        float sn, cs;
        sincosf(6.28318530717958648f * u2, &sn, &cs);
        z[2 * h] = r * cs;
        z[2 * h + 1] = r * sn;
    }
}

// The normal of (token t, expert e) alone (its group's draw, one of the four kept).
__device__ __forceinline__ float routing_noise(int t, int e, uint32_t seed) {
    float z[4];
    routing_noise4(t, e >> 2, seed, z);
    const int j = e & 3;
    return j == 0 ? z[0] : j == 1 ? z[1] : j == 2 ? z[2] : z[3];
}

// ---------------------------------------------------------------- host side
extern std::atomic<uint64_t> g_launches;
inline void count_launch(uint64_t n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Device address of the error word of the current device (cached per device).
int* device_error_word();

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Sub-buffers carved out of the caller's workspace.
struct Workspace {
    char* base;
    size_t used;
    template <typename T> T* take(size_t count) {
        used = align_up(used, 256);
        T* p = reinterpret_cast<T*>(base ? base + used : nullptr);
        used += count * sizeof(T);
        return p;
    }
};

int num_sms();

template <typename V>
inline cudaError_t launch_fill(V* p, long long n, V v, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const long long blocks = std::min<long long>((n + 255) / 256, (long long)num_sms() * 8);
    cudaError_t e = launch_pdl(fill_kernel<V>, dim3((unsigned)blocks), dim3(256), 0, s, p, n, v);
    count_launch();
    return e;
}

}  // namespace moe
