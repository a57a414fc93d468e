// Differentiable balance loss on the soft expert load, and its gradient.
//
// "PyTorch distributed MoE training", section 3.3: balance_loss = mean((load - mean(load))^2)
// on integer counts (no gradient). "Expert Parallelism: Scaling Mixture-of-Experts Models",
// sections 2.2-2.3: the gate probabilities softmax(gate(x) / temperature) and a balance loss
// on the per-expert token fraction. Here the squared-deviation form is applied to the soft
// load P_e = sum_t softmax(z_t / temperature)_e, which makes it differentiable:
//   loss = weight * mean_e (P_e - T/E)^2,   (mean_e P_e = T/E since each softmax sums to 1)
//   g_e = weight * 2 (P_e - T/E) / E,  dz_te = p_te (g_e - sum_j p_tj g_j) / temperature.
// Every reduction runs in a fixed order (warp butterflies, sequential per-thread sums).
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kSoftTok = 64;        // tokens per block of the soft-load partial sums (8 per warp)
constexpr int kSoftThreads = 256;
constexpr int kQ = MOE_MAX_EXPERTS / 32;   // experts per lane (e = lane + 32 q)
constexpr int kDxTok = 8;           // tokens per block of dx += dz Wg
constexpr int kDxThreads = 128;
constexpr int kWgE = 8;             // experts per block of the dz^T x partials
constexpr int kWgThreads = 128;
constexpr int kWgChunk = 32;        // tokens staged in shared memory per round

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One token's probabilities p_e = softmax(z / temp)_e, lane-distributed: p[q] is expert
// lane + 32 q (0 beyond E). The whole warp takes part.
__device__ __forceinline__ void token_softmax(const float* z, int E, float inv_temp, int lane, float (&p)[kQ]) {
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
        const int e = lane + 32 * q;
        p[q] = e < E ? z[e] : -INFINITY;
        mx = fmaxf(mx, p[q]);
    }
    mx = warp_max(mx);
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
        const int e = lane + 32 * q;
        p[q] = e < E ? __expf((p[q] - mx) * inv_temp) : 0.f;
        s += p[q];
    }
    const float inv = 1.f / warp_sum(s);
#pragma unroll
    for (int q = 0; q < kQ; ++q) p[q] *= inv;
}

// Columns [c, c + V) of a row: a 16-byte vector when the row length allows, else guarded
// scalar loads (zero beyond d).
template <typename T>
__device__ __forceinline__ void load_cols(const T* row, int c, int d, float* out) {
    constexpr int V = Vec16<T>::N;
    if ((d % V) == 0) {
        load16(row + c, out);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) out[i] = c + i < d ? ld_f(row + c + i) : 0.f;
    }
}

template <typename T>
__device__ __forceinline__ void store_cols(T* row, int c, int d, const float* in) {
    constexpr int V = Vec16<T>::N;
    if ((d % V) == 0) {
        store16(row + c, in);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (c + i < d) st_f(row + c + i, in[i]);
    }
}

// part[block, e] = sum over the block's 64 tokens of softmax(z_t / temp)_e: each warp sums
// its 8 tokens in order, then the 8 warp sums are added in warp order.
__global__ void __launch_bounds__(kSoftThreads)
soft_load_kernel(const float* __restrict__ logits, int T, int E, float inv_temp, float* __restrict__ part) {
    pdl_wait();
    __shared__ float s_part[kSoftThreads / 32][MOE_MAX_EXPERTS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kSoftTok + warp * (kSoftTok / (kSoftThreads / 32));
    float acc[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) acc[q] = 0.f;
    for (int i = 0; i < kSoftTok / (kSoftThreads / 32); ++i) {
        const int t = t0 + i;
        if (t >= T) break;   // warp-uniform
        float p[kQ];
        token_softmax(logits + (size_t)t * E, E, inv_temp, lane, p);
#pragma unroll
        for (int q = 0; q < kQ; ++q) acc[q] += p[q];
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q)
        if (lane + 32 * q < E) s_part[warp][lane + 32 * q] = acc[q];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSoftThreads / 32; ++w) v += s_part[w][e];
        part[(size_t)blockIdx.x * E + e] = v;
    }
}

// P[e] = sum of the soft-load partials over the chunks: block b takes experts 32 b + lane
// (128-byte rows, coalesced); warp w adds chunks w, w + 32, ..., then the 32 warp sums are
// added in warp order.
constexpr int kFinalThreads = 1024;
__global__ void __launch_bounds__(kFinalThreads)
soft_final_kernel(const float* __restrict__ part, int nchunk, int E, float* __restrict__ P) {
    pdl_wait();
    __shared__ float s_acc[kFinalThreads / 32][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (e < E)
        for (int c = warp; c < nchunk; c += kFinalThreads / 32) acc += part[(size_t)c * E + e];
    s_acc[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && e < E) {
        float v = 0.f;
        for (int w = 0; w < kFinalThreads / 32; ++w) v += s_acc[w][lane];
        P[e] = v;
    }
}

// loss = weight * mean_e (P_e - T/E)^2: one warp, lanes over experts, fixed-order butterfly
// (fp32: GB300's FP64 rate is far too low for a serial loop).
__global__ void __launch_bounds__(32)
soft_loss_kernel(const float* __restrict__ P, int T, int E, float weight, float* __restrict__ loss) {
    pdl_wait();
    const float mean = (float)T / (float)E;
    float s = 0.f;
    for (int e = threadIdx.x; e < E; e += 32) {
        const float dv = P[e] - mean;
        s = fmaf(dv, dv, s);
    }
    s = warp_sum(s);
    if (threadIdx.x == 0) *loss = weight * s / (float)E;
}

// Sum of one value per thread over a block of at most 1024 threads, in a fixed order (warp
// butterflies, then the warp sums in warp order); every thread gets the result.
__device__ __forceinline__ float block_sum(float v) {
    __shared__ float s_w[32];
    __shared__ float s_tot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum(v);
    __syncthreads();   // s_w / s_tot free from a previous call
    if (lane == 0) s_w[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_w[w];
        s_tot = t;
    }
    __syncthreads();
    return s_tot;
}

// Sliding window of soft loads ("Expert Parallelism", section 2.3: load statistics over the
// last batches rather than one). One block, thread e = expert e. state[0] is the ring slot of
// this batch, state[1] the batches already in the window. This batch's P goes into its slot;
// Pbar_e = (sum of the window's n = min(state[1] + 1, W) loads, oldest first) / n;
// loss = weight * mean_e (Pbar_e - mean(Pbar))^2; then the state advances. A state out of
// range records MOE_ERR_DEVICE_BOUNDS and restarts the window.
__global__ void __launch_bounds__(MOE_MAX_EXPERTS)
soft_window_kernel(const float* __restrict__ P, int E, int W, float weight, float* __restrict__ ring,
                   int* __restrict__ state, float* __restrict__ Pbar, float* __restrict__ loss, int* err) {
    pdl_wait();
    __shared__ int s_pos, s_n;
    if (threadIdx.x == 0) {
        int pos = state[0], filled = state[1];
        if (pos < 0 || pos >= W || filled < 0 || filled > W) {
            raise_error(err, kErrBounds);
            pos = 0;
            filled = 0;
        }
        s_pos = pos;
        s_n = min(filled + 1, W);
    }
    __syncthreads();
    const int pos = s_pos, n = s_n, e = threadIdx.x;
    float pb = 0.f;
    if (e < E) {
        const float pe = P[e];
        ring[(size_t)pos * E + e] = pe;
        float acc = 0.f;
        for (int i = n - 1; i >= 1; --i) {   // slots pos - n + 1 .. pos - 1 (mod W): earlier batches
            const int slot = pos - i < 0 ? pos - i + W : pos - i;
            acc += ring[(size_t)slot * E + e];
        }
        pb = (acc + pe) / (float)n;
        Pbar[e] = pb;
    }
    const float mean = block_sum(pb) / (float)E;
    const float dv = e < E ? pb - mean : 0.f;
    const float q = block_sum(dv * dv);
    if (threadIdx.x == 0) {
        if (loss) *loss = weight * q / (float)E;
        state[0] = pos + 1 == W ? 0 : pos + 1;
        state[1] = n;
    }
}

// g_e = weight * 2 (P_e - mean) / E into s_g (every thread of the block calls this). One batch
// (win_n null): mean = T/E exactly, since each token's softmax sums to 1. A window mean load
// (win_n = the window's batch count n): mean = mean_e P_e (fixed order) and g is divided by n,
// the gradient reaching only the current batch's share of the mean.
__device__ __forceinline__ void soft_grad_vector(const float* __restrict__ P, int Tn, int E, float weight,
                                                 const int* __restrict__ win_n, float* s_g) {
    float mean = (float)Tn / (float)E, scale = 1.f;
    if (win_n) {
        float v = 0.f;
        for (int e = threadIdx.x; e < E; e += blockDim.x) v += P[e];
        mean = block_sum(v) / (float)E;
        scale = 1.f / (float)max(1, *win_n);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const float g = weight * 2.f * (P[e] - mean) / (float)E;
        s_g[e] = win_n ? g * scale : g;
    }
    __syncthreads();
}

// For rows that are no multiple of 16 bytes. 8 tokens per block (x), V columns per thread (y).
// dz_te = p_te (g_e - sum_j p_tj g_j) / temp for the block's tokens (written to dz by the first
// column block), then dx[t, c..c+V) += sum_e dz_te Wg[e, c..c+V), experts in ascending order,
// read-modify-write in the activation type.
template <typename T>
__global__ void __launch_bounds__(kDxThreads)
soft_dz_dx_kernel(const float* __restrict__ logits, const float* __restrict__ P, int Tn, int E, int d,
                  float inv_temp, float weight, const int* __restrict__ win_n, const T* __restrict__ Wg,
                  T* __restrict__ dx, float* __restrict__ dz) {
    pdl_wait();
    constexpr int V = Vec16<T>::N;
    __shared__ float s_g[MOE_MAX_EXPERTS];
    __shared__ float s_dz[kDxTok][MOE_MAX_EXPERTS];
    soft_grad_vector(P, Tn, E, weight, win_n, s_g);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kDxTok;
    const int nt = min(kDxTok, Tn - t0);
    for (int i = warp; i < nt; i += kDxThreads / 32) {
        const int t = t0 + i;
        float p[kQ], sdot = 0.f;
        token_softmax(logits + (size_t)t * E, E, inv_temp, lane, p);
#pragma unroll
        for (int q = 0; q < kQ; ++q)
            if (lane + 32 * q < E) sdot += p[q] * s_g[lane + 32 * q];
        sdot = warp_sum(sdot);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int e = lane + 32 * q;
            if (e < E) {
                const float v = p[q] * (s_g[e] - sdot) * inv_temp;
                s_dz[i][e] = v;
                if (blockIdx.y == 0) dz[(size_t)t * E + e] = v;
            }
        }
    }
    __syncthreads();
    const int c = (blockIdx.y * kDxThreads + threadIdx.x) * V;
    if (c >= d) return;
    float acc[kDxTok][V];
#pragma unroll
    for (int i = 0; i < kDxTok; ++i) {
        if (i < nt) load_cols(dx + (size_t)(t0 + i) * d, c, d, acc[i]);
        else {
#pragma unroll
            for (int v = 0; v < V; ++v) acc[i][v] = 0.f;
        }
    }
    // four experts' Wg loads in flight, then their FMAs in ascending expert order
    int e = 0;
    for (; e + 4 <= E; e += 4) {
        float wv[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) load_cols(Wg + (size_t)(e + u) * d, c, d, wv[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < kDxTok; ++i) {
                const float z = s_dz[i][e + u];
#pragma unroll
                for (int v = 0; v < V; ++v) acc[i][v] = fmaf(z, wv[u][v], acc[i][v]);
            }
    }
    for (; e < E; ++e) {
        float wv[V];
        load_cols(Wg + (size_t)e * d, c, d, wv);
#pragma unroll
        for (int i = 0; i < kDxTok; ++i) {
            const float z = s_dz[i][e];
#pragma unroll
            for (int v = 0; v < V; ++v) acc[i][v] = fmaf(z, wv[v], acc[i][v]);
        }
    }
#pragma unroll
    for (int i = 0; i < kDxTok; ++i)
        if (i < nt) store_cols(dx + (size_t)(t0 + i) * d, c, d, acc[i]);
}

// Split-K partials of dz^T x for rows that are no multiple of 16 bytes: part[split, e, c] =
// sum over the split's tokens (in order) of dz[t, e] x[t, c], for 8 experts per block and V
// columns per thread; part[split, e, d] = sum over the split's tokens of dz[t, e] (for dbg),
// from the first column block.
template <typename T>
__global__ void __launch_bounds__(kWgThreads)
soft_dwg_partial_kernel(const float* __restrict__ dz, const T* __restrict__ x, int Tn, int E, int d,
                        int splits, int pitch_, float* __restrict__ part) {
    pdl_wait();
    constexpr int V = Vec16<T>::N;
    __shared__ float s_dz[kWgChunk][kWgE];
    const int e0 = blockIdx.y * kWgE, sp = blockIdx.z;
    const int per = (Tn + splits - 1) / splits;
    const int t0 = sp * per, t1 = min(Tn, t0 + per);
    const int c = (blockIdx.x * kWgThreads + threadIdx.x) * V;
    const bool col_ok = c < d;
    const bool sums = blockIdx.x == 0 && threadIdx.x < kWgE;
    float acc[kWgE][V];
#pragma unroll
    for (int u = 0; u < kWgE; ++u)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[u][v] = 0.f;
    float colsum = 0.f;
    for (int tc = t0; tc < t1; tc += kWgChunk) {
        const int n = min(kWgChunk, t1 - tc);
        __syncthreads();
        for (int j = threadIdx.x; j < kWgChunk * kWgE; j += kWgThreads) {
            const int i = j / kWgE, u = j % kWgE;
            s_dz[i][u] = (i < n && e0 + u < E) ? dz[(size_t)(tc + i) * E + e0 + u] : 0.f;
        }
        __syncthreads();
        if (col_ok) {
            // four token rows in flight, then their FMAs in token order
            int i = 0;
            for (; i + 4 <= n; i += 4) {
                float xv[4][V];
#pragma unroll
                for (int q = 0; q < 4; ++q) load_cols(x + (size_t)(tc + i + q) * d, c, d, xv[q]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int u = 0; u < kWgE; ++u) {
                        const float z = s_dz[i + q][u];
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[u][v] = fmaf(z, xv[q][v], acc[u][v]);
                    }
            }
            for (; i < n; ++i) {
                float xv[V];
                load_cols(x + (size_t)(tc + i) * d, c, d, xv);
#pragma unroll
                for (int u = 0; u < kWgE; ++u) {
                    const float z = s_dz[i][u];
#pragma unroll
                    for (int v = 0; v < V; ++v) acc[u][v] = fmaf(z, xv[v], acc[u][v]);
                }
            }
        }
        if (sums)
            for (int i = 0; i < n; ++i) colsum += s_dz[i][threadIdx.x];
    }
    const size_t pitch = (size_t)pitch_;
#pragma unroll
    for (int u = 0; u < kWgE; ++u) {
        if (e0 + u >= E) break;
        float* row = part + ((size_t)sp * E + e0 + u) * pitch;
#pragma unroll
        for (int v = 0; v < V; ++v)
            if (c + v < d) row[c + v] = acc[u][v];
    }
    if (sums && e0 + threadIdx.x < E) part[((size_t)sp * E + e0 + threadIdx.x) * pitch + d] = colsum;
}

// ---------------------------------------------------------------- tiled kernels (16-byte rows)
// The two contractions of the backward, dx += dz Wg ([T,E] x [E,d]) and dWg += dz^T x
// ([E,T] x [T,d]), on CUDA cores with operand tiles staged in shared memory by cp.async, so
// that many row loads are in flight per SM without holding registers. Each thread owns 8
// consecutive columns and 4 tokens (dx) or 4 experts (dWg).
constexpr int kTileThreads = 256;
constexpr int kTileCols = 512;       // 64 column groups of 8
constexpr int kTileStages = 3;       // dz^T x token pipeline depth

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool pred) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(pred ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 8 consecutive elements at p (16-byte aligned) as floats.
template <typename T>
__device__ __forceinline__ void lds8(const T* p, float* out) {
    if constexpr (sizeof(T) == 2) {
        unpack16<T>(*reinterpret_cast<const uint4*>(p), out);
    } else {
        unpack16<T>(*reinterpret_cast<const uint4*>(p), out);
        unpack16<T>(*reinterpret_cast<const uint4*>(p + 4), out + 4);
    }
}

// dz_te = p_te (g_e - sum_j p_tj g_j) / temp, one warp per token.
__global__ void __launch_bounds__(kSoftThreads)
soft_dz_kernel(const float* __restrict__ logits, const float* __restrict__ P, int Tn, int E, float inv_temp,
               float weight, const int* __restrict__ win_n, float* __restrict__ dz) {
    pdl_wait();
    __shared__ float s_g[MOE_MAX_EXPERTS];
    soft_grad_vector(P, Tn, E, weight, win_n, s_g);
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        float p[kQ], sdot = 0.f;
        token_softmax(logits + (size_t)t * E, E, inv_temp, lane, p);
#pragma unroll
        for (int q = 0; q < kQ; ++q)
            if (lane + 32 * q < E) sdot += p[q] * s_g[lane + 32 * q];
        sdot = warp_sum(sdot);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int e = lane + 32 * q;
            if (e < E) dz[(size_t)t * E + e] = p[q] * (s_g[e] - sdot) * inv_temp;
        }
    }
}

// dx[t, c] += sum_e dz[t, e] Wg[e, c] for 16 tokens (x) x 512 columns (y) per block, experts
// in ascending order. dz of the block's tokens is staged once (transposed: 4 tokens per 16
// bytes); Wg streams through (at most) two stages of ec experts. Shared memory is sized by E:
// E * 64 B + stages * ec * 512 elements.
template <typename T>
__global__ void __launch_bounds__(kTileThreads)
soft_dx_tiled_kernel(const float* __restrict__ dz, const T* __restrict__ Wg, int Tn, int E, int d, int ec,
                     T* __restrict__ dx) {
    pdl_wait();
    constexpr int TB = 16;
    extern __shared__ __align__(16) uint8_t sm[];
    float* zt = reinterpret_cast<float*>(sm);                           // [E][TB]
    T* ws = reinterpret_cast<T*>(sm + (size_t)E * TB * sizeof(float));   // [stages][ec][kTileCols]
    const int tid = threadIdx.x, tc = tid & 63, tt = tid >> 6;
    const int t0 = blockIdx.x * TB;
    const int cb = blockIdx.y * kTileCols;
    const int c = cb + tc * 8;
    const int EC = ec;
    const int nch = (E + EC - 1) / EC;

    auto issue = [&](int ch) {
        T* dst = ws + (size_t)(ch & 1) * EC * kTileCols;
        constexpr int VR = kTileCols * (int)sizeof(T) / 16;   // 16-byte vectors per row
        for (int i = tid; i < EC * VR; i += kTileThreads) {
            const int r = i / VR, v = i % VR;
            const int e = ch * EC + r, cc = cb + v * (16 / (int)sizeof(T));
            const bool ok = e < E && cc < d;
            cp_async16(smem_addr(dst + (size_t)r * kTileCols + v * (16 / (int)sizeof(T))),
                       ok ? (const void*)(Wg + (size_t)e * d + cc) : (const void*)Wg, ok);
        }
    };
    issue(0);
    cp_async_commit();
    for (int i = tid; i < E * TB; i += kTileThreads) {
        const int e = i / TB, r = i % TB;
        zt[i] = t0 + r < Tn ? dz[(size_t)(t0 + r) * E + e] : 0.f;
    }
    float acc[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = 0.f;
        const int t = t0 + tt * 4 + u;
        if (t < Tn && c < d) load_cols(dx + (size_t)t * d, c, d, acc[u]);
        if (sizeof(T) == 4 && t < Tn && c + 4 < d) load_cols(dx + (size_t)t * d, c + 4, d, acc[u] + 4);
    }
    for (int ch = 0; ch < nch; ++ch) {
        if (ch + 1 < nch) issue(ch + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const T* wrow = ws + (size_t)(ch & 1) * EC * kTileCols + tc * 8;
        const int ne = min(EC, E - ch * EC);
        for (int j = 0; j < ne; ++j) {
            float wv[8];
            lds8(wrow + (size_t)j * kTileCols, wv);
            const float4 z = *reinterpret_cast<const float4*>(zt + (size_t)(ch * EC + j) * TB + tt * 4);
            const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(zz[u], wv[v], acc[u][v]);
        }
        __syncthreads();   // the stage is refilled by the next iteration's issue
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = t0 + tt * 4 + u;
        if (t >= Tn || c >= d) continue;
        store_cols(dx + (size_t)t * d, c, d, acc[u]);
        if (sizeof(T) == 4 && c + 4 < d) store_cols(dx + (size_t)t * d, c + 4, d, acc[u] + 4);
    }
}

// Split-K partials of dz^T x for 16 experts (y) x 512 columns (x) per block over a token split
// (z): part[split, e, c] = sum over the split's tokens, in order, of dz[t, e] x[t, c];
// part[split, e, d] = the split's sum of dz[t, e] (for dbg), from the first column block.
// Token chunks of x and dz go through a three-stage cp.async pipeline.
template <typename T>
__global__ void __launch_bounds__(kTileThreads)
soft_dwg_tiled_kernel(const float* __restrict__ dz, const T* __restrict__ x, int Tn, int E, int d, int splits,
                      int pitch, float* __restrict__ part) {
    pdl_wait();
    constexpr int EB = 16;
    constexpr int TS = sizeof(T) == 2 ? 32 : 16;      // 32 KB of x per stage
    constexpr int VR = kTileCols * (int)sizeof(T) / 16;
    extern __shared__ __align__(16) uint8_t sm[];
    T* xs = reinterpret_cast<T*>(sm);                                                   // [S][TS][cols]
    float* zs = reinterpret_cast<float*>(sm + (size_t)kTileStages * TS * kTileCols * sizeof(T));   // [S][TS][EB]
    const int tid = threadIdx.x, tc = tid & 63, te = tid >> 6;
    const int cb = blockIdx.x * kTileCols, e0 = blockIdx.y * EB, sp = blockIdx.z;
    const int per = (Tn + splits - 1) / splits;
    const int t0 = sp * per, t1 = min(Tn, t0 + per);
    const int nch = t1 > t0 ? (t1 - t0 + TS - 1) / TS : 0;
    const int c = cb + tc * 8;
    const bool sums = blockIdx.x == 0 && tid < EB;

    auto issue = [&](int ch) {
        const int st = ch % kTileStages, tb = t0 + ch * TS;
        T* xd = xs + (size_t)st * TS * kTileCols;
        for (int i = tid; i < TS * VR; i += kTileThreads) {
            const int r = i / VR, v = i % VR;
            const int t = tb + r, cc = cb + v * (16 / (int)sizeof(T));
            const bool ok = t < t1 && cc < d;
            cp_async16(smem_addr(xd + (size_t)r * kTileCols + v * (16 / (int)sizeof(T))),
                       ok ? (const void*)(x + (size_t)t * d + cc) : (const void*)x, ok);
        }
        float* zd = zs + (size_t)st * TS * EB;
        for (int i = tid; i < TS * EB; i += kTileThreads) {
            const int r = i / EB, u = i % EB;
            const int t = tb + r, e = e0 + u;
            const bool ok = t < t1 && e < E;
            cp_async4(smem_addr(zd + i), ok ? (const void*)(dz + (size_t)t * E + e) : (const void*)dz, ok);
        }
    };

    float acc[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = 0.f;
    float colsum = 0.f;
#pragma unroll
    for (int ch = 0; ch < kTileStages - 1; ++ch) {
        if (ch < nch) issue(ch);
        cp_async_commit();
    }
    for (int ch = 0; ch < nch; ++ch) {
        cp_async_wait<kTileStages - 2>();
        __syncthreads();   // chunk ch is in place everywhere; chunk ch - 1 is no longer read
        if (ch + kTileStages - 1 < nch) issue(ch + kTileStages - 1);
        cp_async_commit();
        const int st = ch % kTileStages;
        const int n = min(TS, t1 - (t0 + ch * TS));
        const T* xr = xs + (size_t)st * TS * kTileCols + tc * 8;
        const float* zr = zs + (size_t)st * TS * EB + te * 4;
        for (int r = 0; r < n; ++r) {
            float xv[8];
            lds8(xr + (size_t)r * kTileCols, xv);
            const float4 z = *reinterpret_cast<const float4*>(zr + (size_t)r * EB);
            const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[u][v] = fmaf(zz[u], xv[v], acc[u][v]);
        }
        if (sums)
            for (int r = 0; r < n; ++r) colsum += zs[((size_t)st * TS + r) * EB + tid];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = e0 + te * 4 + u;
        if (e >= E) continue;
        float* row = part + ((size_t)sp * E + e) * pitch;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (c + 4 * h < d)
                *reinterpret_cast<float4*>(row + c + 4 * h) =
                    make_float4(acc[u][4 * h], acc[u][4 * h + 1], acc[u][4 * h + 2], acc[u][4 * h + 3]);
    }
    if (sums && e0 + tid < E) part[((size_t)sp * E + e0 + tid) * pitch + d] = colsum;
}

// dWg[e, c] (+)= sum over splits; dbg[e] (+)= the dz column sums. One block per (expert, 32
// columns): warp w adds splits w, w + 8, ... in order, then the 8 warp sums are added in
// warp order.
__global__ void __launch_bounds__(kSoftThreads)
soft_dwg_reduce_kernel(const float* __restrict__ part, int E, int d, int splits, int pitch_, bool accumulate,
                       float* __restrict__ dWg, float* __restrict__ dbg) {
    pdl_wait();
    __shared__ float s_acc[kSoftThreads / 32][32];
    const int e = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 32 + lane;
    const size_t pitch = (size_t)pitch_;
    float acc = 0.f;
    if (c <= d) {
#pragma unroll 4
        for (int sp = warp; sp < splits; sp += kSoftThreads / 32) acc += part[((size_t)sp * E + e) * pitch + c];
    }
    s_acc[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c <= d) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSoftThreads / 32; ++w) v += s_acc[w][lane];
        if (c < d) dWg[(size_t)e * d + c] = accumulate ? dWg[(size_t)e * d + c] + v : v;
        else if (dbg) dbg[e] = accumulate ? dbg[e] + v : v;
    }
}

// ---------------------------------------------------------------- tensor-core contractions
// dz is fp32; the tcgen05 GEMMs take bf16. Each value is split into hi = bf16(dz) and
// lo = bf16(dz - hi), so hi + lo carries about 16 significant bits, and
//   dz Wg  = [hi | lo] [Wg ; Wg]        (K = 2 E, padded)
//   dz^T x = hi^T x + lo^T x            (rows E8 + e of the product hold lo^T x)
// with every product of bf16 values exact in the fp32 accumulators.
constexpr int kSplitThreads = 256;

__host__ __device__ inline int e8_of(int E) { return (E + 7) / 8 * 8; }
__host__ __device__ inline int k2_of(int E) { return (2 * e8_of(E) + 63) / 64 * 64; }

// dzs[t, c] for t < T_pad, c < K2: hi of dz[t, c] (c < E), lo of dz[t, c - E8]
// (E8 <= c < E8 + E), 0 elsewhere and for t >= T. One thread per 8-column group of a row (the
// groups never straddle a region boundary, since E8 is a multiple of 8; one 16-byte store),
// grid-stride, with 32-bit index arithmetic when the element count allows. Block 0 also
// writes the bucket offsets. (A 64-bit division per column pair had made the kernel 31 us at
// 32768 x 256.)
__device__ __forceinline__ void split_group(const float* __restrict__ dz, int Tn, int E, int e8, int k2, int t,
                                            int c, __nv_bfloat16* __restrict__ dzs) {
    float v[8];
    const bool lo = c >= e8;
    const int src = lo ? c - e8 : c;   // first dz column of the group
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const bool live = t < Tn && src + j < E && (lo ? c < e8 + E : true);
        const float z = live ? dz[(size_t)t * E + src + j] : 0.f;
        const float hi = __bfloat162float(__float2bfloat16_rn(z));
        v[j] = lo ? z - hi : hi;
    }
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    *reinterpret_cast<uint4*>(dzs + (size_t)t * k2 + c) = u;
}

__global__ void __launch_bounds__(kSplitThreads)
soft_split_kernel(const float* __restrict__ dz, int Tn, int Tpad, int E, __nv_bfloat16* __restrict__ dzs,
                  int32_t* __restrict__ offs, int splits, int bucket) {
    pdl_wait();
    const int e8 = e8_of(E), k2 = k2_of(E), groups = k2 / 8;
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= splits; i += blockDim.x) offs[i] = min(i * bucket, Tpad);
        if (threadIdx.x == 0) { offs[splits + 1] = 0; offs[splits + 2] = Tpad; }
    }
    const long long n = (long long)Tpad * groups;
    if (n <= 0x7fffffffLL - (long long)gridDim.x * blockDim.x) {
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < (int)n; i += gridDim.x * blockDim.x) {
            const int t = i / groups;
            split_group(dz, Tn, E, e8, k2, t, (i - t * groups) * 8, dzs);
        }
    } else {
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
            const int t = (int)(i / groups);
            split_group(dz, Tn, E, e8, k2, t, (int)(i - (long long)t * groups) * 8, dzs);
        }
    }
}

// dbg_part[b, e] = sum of dz[t, e] over the 64 rows of block b (in order), thread e.
constexpr int kDzsumRows = 64;
__global__ void __launch_bounds__(256)
soft_dzsum_kernel(const float* __restrict__ dz, int Tn, int E, float* __restrict__ dbg_part) {
    pdl_wait();
    const int t0 = blockIdx.x * kDzsumRows, t1 = min(Tn, t0 + kDzsumRows);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float a = 0.f;
        for (int t = t0; t < t1; ++t) a += dz[(size_t)t * E + e];
        dbg_part[(size_t)blockIdx.x * E + e] = a;
    }
}

// wge[r, c] = Wg[r, c] for r < E, Wg[r - E8, c] for E8 <= r < E8 + E, 0 otherwise.
__global__ void __launch_bounds__(256)
soft_wge_kernel(const __nv_bfloat16* __restrict__ Wg, int E, int d, __nv_bfloat16* __restrict__ wge) {
    pdl_wait();
    const int e8 = e8_of(E), k2 = k2_of(E);
    const long long n = (long long)k2 * d;
    const long long stride = (long long)gridDim.x * blockDim.x;
    if (n + stride <= 0x7fffffffLL) {
        // 32-bit index arithmetic (a 64-bit division per item is a long software sequence)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < (int)n; i += (int)stride) {
            const int r = i / d, c = i - r * d;
            const int src = r < E ? r : (r >= e8 && r < e8 + E ? r - e8 : -1);
            wge[i] = src >= 0 ? Wg[(size_t)src * d + c] : __float2bfloat16_rn(0.f);
        }
    } else {
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
            const int r = (int)(i / d), c = (int)(i % d);
            const int src = r < E ? r : (r >= e8 && r < e8 + E ? r - e8 : -1);
            wge[i] = src >= 0 ? Wg[(size_t)src * d + c] : __float2bfloat16_rn(0.f);
        }
    }
}

// dWg[e, c] (+)= sum over splits (in order) of wpart[s, e, c] + wpart[s, E8 + e, c];
// dbg[e] (+)= sum over blocks (in order) of dbg_part[b, e] (block x = 0, one warp per expert).
__global__ void __launch_bounds__(256)
soft_dwg_tc_reduce_kernel(const float* __restrict__ wpart, int splits, int E, int d, const float* __restrict__ dbg_part,
                          int nblk, bool accumulate, float* __restrict__ dWg, float* __restrict__ dbg) {
    pdl_wait();
    const int e = blockIdx.y;
    const int e8 = e8_of(E), k2 = k2_of(E);
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < d) {
        float v = 0.f;
        for (int sp = 0; sp < splits; ++sp) {
            const float* base = wpart + (size_t)sp * k2 * d;
            v += base[(size_t)e * d + c] + base[(size_t)(e8 + e) * d + c];
        }
        dWg[(size_t)e * d + c] = accumulate ? dWg[(size_t)e * d + c] + v : v;
    }
    if (blockIdx.x == 0 && threadIdx.x < 32 && dbg) {
        const int lane = threadIdx.x;
        float a = 0.f;
        for (int b = lane; b < nblk; b += 32) a += dbg_part[(size_t)b * E + e];
        a = warp_sum(a);
        if (lane == 0) dbg[e] = accumulate ? dbg[e] + a : a;
    }
}

}  // namespace

int soft_chunks(const moe_config_t& c) { return std::max(1, ceil_div(c.T, kSoftTok)); }

static int dwg_col_blocks(const moe_config_t& c) {
    const int V = c.dtype == MOE_BF16 ? 8 : 4;
    return std::max(1, ceil_div(c.d, kWgThreads * V));
}

// Row pitch of the dz^T x partials: d columns + the dz column sum, rounded up to 16 bytes.
static int dwg_pitch(const moe_config_t& c) { return (c.d + 1 + 3) / 4 * 4; }

int soft_splits(const moe_config_t& c) {
    // about two blocks of the tiled kernel per SM; each split covers at least 16 tokens
    const long long blocks = (long long)ceil_div(c.d, kTileCols) * ceil_div(c.E, 16);
    const int s = (int)std::min<long long>(256, ceil_div(2LL * num_sms(), blocks));
    const int cap = std::max(1, ceil_div(c.T, 16));
    return std::max(1, std::min(s, cap));
}

// The tiled kernels need rows of whole 16-byte vectors and 16-byte aligned bases.
static bool tiled_ok(const moe_config_t& c, const void* a, const void* b) {
    const int V = c.dtype == MOE_BF16 ? 8 : 4;
    return c.d % V == 0 && (((uintptr_t)a | (uintptr_t)b) & 15) == 0;
}

// experts per Wg stage of soft_dx_tiled_kernel (32 KB per stage at most) and its shared memory
template <typename T>
static int dx_tiled_ec(int E) { return std::min(E, sizeof(T) == 2 ? 32 : 16); }
template <typename T>
static size_t dx_tiled_smem(int E) {
    const int ec = dx_tiled_ec<T>(E);
    const int stages = E > ec ? 2 : 1;
    return (size_t)E * 16 * sizeof(float) + (size_t)stages * ec * kTileCols * sizeof(T);
}
template <typename T>
static size_t dwg_tiled_smem() {
    constexpr int TS = sizeof(T) == 2 ? 32 : 16;
    return (size_t)kTileStages * TS * (kTileCols * sizeof(T) + 16 * sizeof(float));
}

// Tensor cores from 32 experts up; below that the contractions are a few FMAs per loaded
// element and the tiled CUDA-core kernels take as long with fewer launches (measured equal at
// 8192 x 16).
bool soft_tc_ok(const moe_config_t& c) { return c.dtype == MOE_BF16 && c.d % 64 == 0 && c.E >= 32; }

// Geometry of the tensor-core contractions: tokens padded to the 256-row tiles, and the
// token buckets (split-K) of dz^T x, sized so that about one round of CTA pairs is busy.
struct SoftTc {
    int tpad, k2, splits, bucket, nblk;
};
static SoftTc soft_tc_geom(const moe_config_t& c) {
    SoftTc g;
    g.tpad = std::max(256, (c.T + 255) / 256 * 256);
    g.k2 = k2_of(c.E);
    const long long tiles_per_split = (long long)ceil_div(g.k2, 256) * ceil_div(c.d, 256);
    const int want = (int)std::max<long long>(1, (num_sms() / 2 + tiles_per_split - 1) / tiles_per_split);
    const int max_splits = std::max(1, g.tpad / 256);   // buckets of at least 256 rows
    g.splits = std::min(want, max_splits);
    g.bucket = (ceil_div(g.tpad, g.splits) + 63) / 64 * 64;
    g.splits = ceil_div(g.tpad, g.bucket);
    g.nblk = std::max(1, ceil_div(c.T, kDzsumRows));   // dz column-sum partials
    return g;
}

void soft_scratch_take(Workspace& ws, const moe_config_t& c, SoftScratch* s) {
    s->part = ws.take<float>((size_t)soft_chunks(c) * c.E);
    s->dz = ws.take<float>((size_t)c.T * c.E + 1);
    s->dwg_part = ws.take<float>((size_t)soft_splits(c) * c.E * dwg_pitch(c));
    if (soft_tc_ok(c)) {
        const SoftTc g = soft_tc_geom(c);
        s->dzs = ws.take<__nv_bfloat16>((size_t)g.tpad * g.k2);
        s->wge = ws.take<__nv_bfloat16>((size_t)g.k2 * c.d);
        s->offs = ws.take<int32_t>((size_t)g.splits + 3);
        s->wpart = ws.take<float>((size_t)g.splits * g.k2 * c.d);
        s->dbg_part = ws.take<float>((size_t)g.nblk * c.E);
    } else {
        s->dzs = s->wge = nullptr;
        s->offs = nullptr;
        s->wpart = s->dbg_part = nullptr;
    }
}

// dz (fp32 [T, E]) -> hi/lo bf16 layout and bucket offsets; with want_sums also the column-sum
// partials of dz (for dbg).
static cudaError_t launch_soft_split(const moe_config_t& c, const float* dz, bool want_sums, const SoftScratch& s,
                                     cudaStream_t st) {
    const SoftTc g = soft_tc_geom(c);
    const long long n = (long long)g.tpad * (g.k2 / 8);
    const int grid = (int)std::max(1LL, std::min((n + kSplitThreads - 1) / kSplitThreads, (long long)num_sms() * 8));
    cudaError_t e = launch_pdl(soft_split_kernel, dim3(grid), dim3(kSplitThreads), 0, st, dz, c.T, g.tpad, c.E,
                               (__nv_bfloat16*)s.dzs, s.offs, g.splits, g.bucket);
    count_launch();
    if (e != cudaSuccess || !want_sums || c.T == 0) return e;
    e = launch_pdl(soft_dzsum_kernel, dim3(g.nblk), dim3(256), 0, st, dz, c.T, c.E, s.dbg_part);
    count_launch();
    return e;
}

// dWg (+)= dz^T x, dbg (+)= column sums of dz, from the split layout already in s.dzs.
static cudaError_t launch_dzx_tc(const moe_config_t& c, const void* x, float* dWg, float* dbg, bool accumulate,
                                 const SoftScratch& s, cudaStream_t st) {
    const SoftTc g = soft_tc_geom(c);
    WgradArgs wa{s.dzs, x, s.wpart, s.offs, g.splits, g.k2, c.d};
    wa.rows_p = g.tpad;
    wa.rows_q = std::max(c.T, 1);
    wa.f32 = true;
    cudaError_t e = launch_wgrad_tc_pair(c, wa, st);
    if (e != cudaSuccess) return e;
    dim3 gr(ceil_div(c.d, 256), c.E);
    e = launch_pdl(soft_dwg_tc_reduce_kernel, gr, dim3(256), 0, st, (const float*)s.wpart, g.splits, c.E, c.d,
                   (const float*)s.dbg_part, g.nblk, accumulate, dWg, dbg);
    count_launch();
    return e;
}

// dx += dz Wg from the split layout already in s.dzs.
static cudaError_t launch_dzwg_tc(const moe_config_t& c, const void* Wg, void* dx, const SoftScratch& s,
                                  cudaStream_t st) {
    const SoftTc g = soft_tc_geom(c);
    const long long n = (long long)g.k2 * c.d;
    const int grid = (int)std::min<long long>((n + 255) / 256, (long long)num_sms() * 8);
    cudaError_t e = launch_pdl(soft_wge_kernel, dim3(grid), dim3(256), 0, st, (const __nv_bfloat16*)Wg, c.E, c.d,
                               (__nv_bfloat16*)s.wge);
    count_launch();
    if (e != cudaSuccess) return e;
    RowGemmArgs ra{};
    ra.kind = kGemmAccum;
    ra.A = s.dzs; ra.B = s.wge; ra.aux = dx; ra.out0 = dx;
    ra.offsets = s.offs + g.splits + 1;   // one bucket [0, T_pad]
    ra.E = 1; ra.N = c.d; ra.K = g.k2; ra.rows_capacity = g.tpad;
    ra.sBe = 0; ra.sBn = 1; ra.sBk = c.d;
    ra.rows_valid = c.T;
    return launch_row_gemm_tc_pair(c, ra, st);
}

cudaError_t launch_soft_balance(const moe_config_t& c, const float* logits, float weight, float* P,
                                float* loss, const SoftScratch& s, cudaStream_t st) {
    const float inv_temp = 1.0f / c.temperature;
    const int nchunk = soft_chunks(c);
    if (c.T > 0) {
        launch_pdl(soft_load_kernel, nchunk, kSoftThreads, 0, st, logits, c.T, c.E, inv_temp, s.part);
        count_launch();
    } else {
        cudaError_t e = launch_fill(s.part, (long long)c.E, 0.f, st);
        if (e != cudaSuccess) return e;
    }
    launch_pdl(soft_final_kernel, ceil_div(c.E, 32), kFinalThreads, 0, st, s.part, nchunk, c.E, P);
    count_launch();
    if (loss) {
        launch_pdl(soft_loss_kernel, 1, 32, 0, st, (const float*)P, c.T, c.E, weight, loss);
        count_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_soft_window(const moe_config_t& c, const float* P, float weight, int W, float* ring,
                               int32_t* state, float* Pbar, float* loss, cudaStream_t st) {
    launch_pdl(soft_window_kernel, 1, MOE_MAX_EXPERTS, 0, st, P, c.E, W, weight, ring, (int*)state, Pbar, loss,
               device_error_word());
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_soft_balance_bwd(const moe_config_t& c, const float* logits, const float* P, float weight,
                                    const int32_t* win_n, const void* x, const void* Wg, void* dx, float* dWg,
                                    float* dbg, const SoftScratch& s, cudaStream_t st) {
    if (c.T == 0) return cudaSuccess;
    const float inv_temp = 1.0f / c.temperature;
    if (soft_tc_ok(c)) {
        // dz on CUDA cores, both contractions on the tensor cores
        const int g0 = std::max(1, std::min(ceil_div(c.T, kSoftThreads / 32), num_sms() * 8));
        cudaError_t e = launch_pdl(soft_dz_kernel, dim3(g0), dim3(kSoftThreads), 0, st, logits, P, c.T, c.E,
                                   inv_temp, weight, (const int*)win_n, s.dz);
        count_launch();
        if (e != cudaSuccess) return e;
        if ((e = launch_soft_split(c, s.dz, dbg != nullptr, s, st)) != cudaSuccess) return e;
        if ((e = launch_dzwg_tc(c, Wg, dx, s, st)) != cudaSuccess) return e;
        return launch_dzx_tc(c, x, dWg, dbg, true, s, st);
    }
    if (tiled_ok(c, Wg, dx)) {
        const int g0 = std::max(1, std::min(ceil_div(c.T, kSoftThreads / 32), num_sms() * 8));
        launch_pdl(soft_dz_kernel, g0, kSoftThreads, 0, st, logits, P, c.T, c.E, inv_temp, weight,
                   (const int*)win_n, s.dz);
        count_launch();
        dim3 g(ceil_div(c.T, 16), ceil_div(c.d, kTileCols));
        if (c.dtype == MOE_BF16) {
            auto k = soft_dx_tiled_kernel<__nv_bfloat16>;
            const size_t sm = dx_tiled_smem<__nv_bfloat16>(c.E);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e != cudaSuccess) return e;
            launch_pdl(k, g, kTileThreads, sm, st, s.dz, (const __nv_bfloat16*)Wg, c.T, c.E, c.d,
                                           dx_tiled_ec<__nv_bfloat16>(c.E), (__nv_bfloat16*)dx);
        } else {
            auto k = soft_dx_tiled_kernel<float>;
            const size_t sm = dx_tiled_smem<float>(c.E);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e != cudaSuccess) return e;
            launch_pdl(k, g, kTileThreads, sm, st, s.dz, (const float*)Wg, c.T, c.E, c.d, dx_tiled_ec<float>(c.E),
                                           (float*)dx);
        }
        count_launch();
    } else {
        const int V = c.dtype == MOE_BF16 ? 8 : 4;
        dim3 g0(ceil_div(c.T, kDxTok), ceil_div(c.d, kDxThreads * V));
        if (c.dtype == MOE_BF16)
            launch_pdl(soft_dz_dx_kernel<__nv_bfloat16>, g0, kDxThreads, 0, st, logits, P, c.T, c.E, c.d, inv_temp,
                       weight, (const int*)win_n, (const __nv_bfloat16*)Wg, (__nv_bfloat16*)dx, s.dz);
        else
            launch_pdl(soft_dz_dx_kernel<float>, g0, kDxThreads, 0, st, logits, P, c.T, c.E, c.d, inv_temp, weight,
                       (const int*)win_n, (const float*)Wg, (float*)dx, s.dz);
        count_launch();
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_dense_dwg(c, s.dz, x, dWg, dbg, true, s, st);
}

cudaError_t launch_dense_dwg(const moe_config_t& c, const float* dz, const void* x, float* dWg, float* dbg,
                             bool accumulate, const SoftScratch& s, cudaStream_t st) {
    if (c.T == 0 && accumulate) return cudaSuccess;
    if (c.T > 0 && soft_tc_ok(c)) {
        cudaError_t e = launch_soft_split(c, dz, dbg != nullptr, s, st);
        if (e != cudaSuccess) return e;
        return launch_dzx_tc(c, x, dWg, dbg, accumulate, s, st);
    }
    const int splits = soft_splits(c);
    const int pitch = dwg_pitch(c);
    if (c.T > 0 && tiled_ok(c, x, s.dwg_part)) {
        dim3 g1(ceil_div(c.d, kTileCols), ceil_div(c.E, 16), splits);
        if (c.dtype == MOE_BF16) {
            auto k = soft_dwg_tiled_kernel<__nv_bfloat16>;
            const size_t sm = dwg_tiled_smem<__nv_bfloat16>();
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e != cudaSuccess) return e;
            launch_pdl(k, g1, kTileThreads, sm, st, dz, (const __nv_bfloat16*)x, c.T, c.E, c.d, splits, pitch, s.dwg_part);
        } else {
            auto k = soft_dwg_tiled_kernel<float>;
            const size_t sm = dwg_tiled_smem<float>();
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
            if (e != cudaSuccess) return e;
            launch_pdl(k, g1, kTileThreads, sm, st, dz, (const float*)x, c.T, c.E, c.d, splits, pitch, s.dwg_part);
        }
        count_launch();
    } else if (c.T > 0) {
        dim3 g1(dwg_col_blocks(c), ceil_div(c.E, kWgE), splits);
        if (c.dtype == MOE_BF16)
            launch_pdl(soft_dwg_partial_kernel<__nv_bfloat16>, g1, kWgThreads, 0, st, dz, (const __nv_bfloat16*)x, c.T,
                                                                             c.E, c.d, splits, pitch, s.dwg_part);
        else
            launch_pdl(soft_dwg_partial_kernel<float>, g1, kWgThreads, 0, st, dz, (const float*)x, c.T, c.E, c.d,
                                                                     splits, pitch, s.dwg_part);
        count_launch();
    } else {
        cudaError_t e = launch_fill(s.dwg_part, (long long)splits * c.E * pitch, 0.f, st);
        if (e != cudaSuccess) return e;
    }
    dim3 g2(ceil_div(c.d + 1, 32), c.E);
    launch_pdl(soft_dwg_reduce_kernel, g2, kSoftThreads, 0, st, s.dwg_part, c.E, c.d, splits, pitch, accumulate, dWg, dbg);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
