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

constexpr int kSoftTok = 64;      // tokens per chunk of the soft-load partial sums
constexpr int kSoftThreads = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One token's softmax normaliser: m = max_e z_e, inv = 1 / sum_e exp((z_e - m) / temp).
__device__ __forceinline__ void token_softmax_stats(const float* z, int E, float inv_temp, int lane,
                                                    float& m, float& inv) {
    float mx = -INFINITY;
    for (int e = lane; e < E; e += 32) mx = fmaxf(mx, z[e]);
    mx = warp_max(mx);
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += __expf((z[e] - mx) * inv_temp);
    s = warp_sum(s);
    m = mx;
    inv = 1.f / s;
}

// part[chunk, e] = sum over the chunk's tokens (in order) of softmax(z_t / temp)_e.
__global__ void __launch_bounds__(kSoftThreads)
soft_load_kernel(const float* __restrict__ logits, int T, int E, float inv_temp, float* __restrict__ part) {
    __shared__ float s_m[kSoftTok], s_inv[kSoftTok];
    const int t0 = blockIdx.x * kSoftTok;
    const int nt = min(kSoftTok, T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < nt; i += kSoftThreads / 32) {
        float m, inv;
        token_softmax_stats(logits + (size_t)(t0 + i) * E, E, inv_temp, lane, m, inv);
        if (lane == 0) { s_m[i] = m; s_inv[i] = inv; }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.f;
        for (int i = 0; i < nt; ++i) acc += __expf((logits[(size_t)(t0 + i) * E + e] - s_m[i]) * inv_temp) * s_inv[i];
        part[(size_t)blockIdx.x * E + e] = acc;
    }
}

// P[e] = sum over chunks (in order); loss = weight * mean_e (P_e - T/E)^2 in double.
__global__ void __launch_bounds__(kSoftThreads)
soft_final_kernel(const float* __restrict__ part, int nchunk, int T, int E, float weight,
                  float* __restrict__ P, float* __restrict__ loss) {
    __shared__ float s_P[MOE_MAX_EXPERTS];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.f;
        for (int c = 0; c < nchunk; ++c) acc += part[(size_t)c * E + e];
        s_P[e] = acc;
        P[e] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0 && loss) {
        const double mean = (double)T / (double)E;
        double s = 0.0;
        for (int e = 0; e < E; ++e) {
            const double dv = (double)s_P[e] - mean;
            s += dv * dv;
        }
        *loss = (float)((double)weight * s / (double)E);
    }
}

// Per token (one warp): dz_te = p_te (g_e - sum_j p_tj g_j) / temp, written to dz, and
// dx[t] += sum_e dz_te Wg[e] (read-modify-write in the activation type).
template <typename T>
__global__ void __launch_bounds__(kSoftThreads)
soft_dz_kernel(const float* __restrict__ logits, const float* __restrict__ P, int Tn, int E, int d,
               float inv_temp, float weight, const T* __restrict__ Wg, T* __restrict__ dx,
               float* __restrict__ dz) {
    __shared__ float s_g[MOE_MAX_EXPERTS];
    const float mean = (float)Tn / (float)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_g[e] = weight * 2.f * (P[e] - mean) / (float)E;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        const float* z = logits + (size_t)t * E;
        float m, inv;
        token_softmax_stats(z, E, inv_temp, lane, m, inv);
        float pe[MOE_MAX_EXPERTS / 32], sdot = 0.f;
#pragma unroll
        for (int q = 0; q < MOE_MAX_EXPERTS / 32; ++q) {
            const int e = lane + 32 * q;
            pe[q] = e < E ? __expf((z[e] - m) * inv_temp) * inv : 0.f;
            sdot += e < E ? pe[q] * s_g[e] : 0.f;
        }
        sdot = warp_sum(sdot);
        float dzl[MOE_MAX_EXPERTS / 32];
#pragma unroll
        for (int q = 0; q < MOE_MAX_EXPERTS / 32; ++q) {
            const int e = lane + 32 * q;
            dzl[q] = e < E ? pe[q] * (s_g[e] - sdot) * inv_temp : 0.f;
            if (e < E) dz[(size_t)t * E + e] = dzl[q];
        }
        if ((d % V) == 0) {
            // warp-uniform trip count: every lane takes part in the shuffles
            for (int c0 = 0; c0 < d; c0 += 32 * V) {
                const int c = c0 + lane * V;
                const bool active = c < d;
                float acc[V];
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = 0.f;
                if (active) load16(dx + (size_t)t * d + c, acc);
                for (int e = 0; e < E; ++e) {
                    float dze = 0.f;
#pragma unroll
                    for (int q = 0; q < MOE_MAX_EXPERTS / 32; ++q)
                        if (q == (e >> 5)) dze = __shfl_sync(0xffffffffu, dzl[q], e & 31);
                    if (active) {
                        float wv[V];
                        load16(Wg + (size_t)e * d + c, wv);
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[i] = fmaf(dze, wv[i], acc[i]);
                    }
                }
                if (active) store16(dx + (size_t)t * d + c, acc);
            }
        } else {
            for (int c0 = 0; c0 < d; c0 += 32) {
                const int c = c0 + lane;
                float acc = c < d ? ld_f(dx + (size_t)t * d + c) : 0.f;
                for (int e = 0; e < E; ++e) {
                    float dze = 0.f;
#pragma unroll
                    for (int q = 0; q < MOE_MAX_EXPERTS / 32; ++q)
                        if (q == (e >> 5)) dze = __shfl_sync(0xffffffffu, dzl[q], e & 31);
                    if (c < d) acc = fmaf(dze, ld_f(Wg + (size_t)e * d + c), acc);
                }
                if (c < d) st_f(dx + (size_t)t * d + c, acc);
            }
        }
    }
}

// Split-K partials of dz^T x: part[split, e, c] = sum over the split's tokens (in order) of
// dz[t, e] * x[t, c]; split column c == d holds sum_t dz[t, e] (for dbg).
template <typename T>
__global__ void __launch_bounds__(kSoftThreads)
soft_dwg_partial_kernel(const float* __restrict__ dz, const T* __restrict__ x, int Tn, int E, int d,
                        int splits, float* __restrict__ part) {
    const int e = blockIdx.y, sp = blockIdx.z;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c > d) return;
    const int per = (Tn + splits - 1) / splits;
    const int t0 = sp * per, t1 = min(Tn, t0 + per);
    // four independent accumulators (tokens t0+4i+u), summed in a fixed order at the end, so
    // that four row loads are in flight per thread
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int t = t0;
    if (c < d) {
        for (; t + 4 <= t1; t += 4) {
            const float z0 = dz[(size_t)t * E + e], z1 = dz[(size_t)(t + 1) * E + e];
            const float z2 = dz[(size_t)(t + 2) * E + e], z3 = dz[(size_t)(t + 3) * E + e];
            const float x0 = ld_f(x + (size_t)t * d + c), x1 = ld_f(x + (size_t)(t + 1) * d + c);
            const float x2 = ld_f(x + (size_t)(t + 2) * d + c), x3 = ld_f(x + (size_t)(t + 3) * d + c);
            a0 = fmaf(z0, x0, a0); a1 = fmaf(z1, x1, a1); a2 = fmaf(z2, x2, a2); a3 = fmaf(z3, x3, a3);
        }
        for (; t < t1; ++t) a0 = fmaf(dz[(size_t)t * E + e], ld_f(x + (size_t)t * d + c), a0);
    } else {
        for (; t + 4 <= t1; t += 4) {
            a0 += dz[(size_t)t * E + e]; a1 += dz[(size_t)(t + 1) * E + e];
            a2 += dz[(size_t)(t + 2) * E + e]; a3 += dz[(size_t)(t + 3) * E + e];
        }
        for (; t < t1; ++t) a0 += dz[(size_t)t * E + e];
    }
    part[((size_t)sp * E + e) * (d + 1) + c] = (a0 + a1) + (a2 + a3);
}

// dWg[e, c] += sum over splits (in order); dbg[e] += the dz column sums.
__global__ void __launch_bounds__(kSoftThreads)
soft_dwg_reduce_kernel(const float* __restrict__ part, int E, int d, int splits, float* __restrict__ dWg,
                       float* __restrict__ dbg) {
    const int e = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c > d) return;
    float acc = 0.f;
    for (int sp = 0; sp < splits; ++sp) acc += part[((size_t)sp * E + e) * (d + 1) + c];
    if (c < d) dWg[(size_t)e * d + c] += acc;
    else if (dbg) dbg[e] += acc;
}

}  // namespace

int soft_chunks(const moe_config_t& c) { return std::max(1, ceil_div(c.T, kSoftTok)); }

int soft_splits(const moe_config_t& c) {
    const int col_blocks = ceil_div(c.d + 1, kSoftThreads);
    // enough blocks for ~16 per SM; each split covers at least 64 tokens
    const int s = ceil_div(16LL * num_sms(), (long long)c.E * col_blocks);
    const int cap = std::max(1, ceil_div(c.T, 64));
    return std::max(1, std::min(std::min(s, 256), cap));
}

void soft_scratch_take(Workspace& ws, const moe_config_t& c, SoftScratch* s) {
    s->part = ws.take<float>((size_t)soft_chunks(c) * c.E);
    s->dz = ws.take<float>((size_t)c.T * c.E + 1);
    s->dwg_part = ws.take<float>((size_t)soft_splits(c) * c.E * (c.d + 1));
}

cudaError_t launch_soft_balance(const moe_config_t& c, const float* logits, float weight, float* P,
                                float* loss, const SoftScratch& s, cudaStream_t st) {
    const float inv_temp = 1.0f / c.temperature;
    const int nchunk = soft_chunks(c);
    if (c.T > 0) {
        soft_load_kernel<<<nchunk, kSoftThreads, 0, st>>>(logits, c.T, c.E, inv_temp, s.part);
        count_launch();
    } else {
        cudaError_t e = cudaMemsetAsync(s.part, 0, sizeof(float) * c.E, st);
        if (e != cudaSuccess) return e;
    }
    soft_final_kernel<<<1, kSoftThreads, 0, st>>>(s.part, nchunk, c.T, c.E, weight, P, loss);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_soft_balance_bwd(const moe_config_t& c, const float* logits, const float* P, float weight,
                                    const void* x, const void* Wg, void* dx, float* dWg, float* dbg,
                                    const SoftScratch& s, cudaStream_t st) {
    if (c.T == 0) return cudaSuccess;
    const float inv_temp = 1.0f / c.temperature;
    const int grid = std::max(1, std::min(ceil_div(c.T, kSoftThreads / 32), num_sms() * 8));
    if (c.dtype == MOE_BF16)
        soft_dz_kernel<__nv_bfloat16><<<grid, kSoftThreads, 0, st>>>(
            logits, P, c.T, c.E, c.d, inv_temp, weight, (const __nv_bfloat16*)Wg, (__nv_bfloat16*)dx, s.dz);
    else
        soft_dz_kernel<float><<<grid, kSoftThreads, 0, st>>>(logits, P, c.T, c.E, c.d, inv_temp, weight,
                                                             (const float*)Wg, (float*)dx, s.dz);
    count_launch();
    const int splits = soft_splits(c);
    dim3 g1(ceil_div(c.d + 1, kSoftThreads), c.E, splits);
    if (c.dtype == MOE_BF16)
        soft_dwg_partial_kernel<__nv_bfloat16><<<g1, kSoftThreads, 0, st>>>(s.dz, (const __nv_bfloat16*)x, c.T,
                                                                           c.E, c.d, splits, s.dwg_part);
    else
        soft_dwg_partial_kernel<float><<<g1, kSoftThreads, 0, st>>>(s.dz, (const float*)x, c.T, c.E, c.d,
                                                                   splits, s.dwg_part);
    count_launch();
    dim3 g2(ceil_div(c.d + 1, kSoftThreads), c.E);
    soft_dwg_reduce_kernel<<<g2, kSoftThreads, 0, st>>>(s.dwg_part, c.E, c.d, splits, dWg, dbg);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
