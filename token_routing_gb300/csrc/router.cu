// Router: gate linear (fp32 accumulation) + top-k (ties -> lower expert id) + softmax over
// the k selected logits divided by the temperature + expert counts, and the balance loss.
//
// "Native MoE training system PithTrain", section 4.1 (gate = Linear(dim, num_experts),
// torch.topk(logits, k) then softmax over the selected values); "Expert Parallelism: Scaling
// Mixture-of-Experts Models", section 2.2 (softmax(gate(x) / temperature), top-8
// pre-selection) and section 5.5 (routing kept in FP32); "PyTorch distributed MoE training",
// section 3.3 (balance_loss = mean((load - mean(load))^2)).
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kRouteTok = 32;     // tokens per block
constexpr int kRouteKc = 32;      // d-chunk staged in shared memory
constexpr int kRouteThreads = 256;
constexpr int kNoExpert = 0x7fffffff;

// (v1, e1) ranks before (v2, e2): larger logit first, lower expert id among equal logits;
// any real candidate ranks before the empty one.
__device__ __forceinline__ bool beats(float v1, int e1, float v2, int e2) {
    if (e1 == kNoExpert) return false;
    if (e2 == kNoExpert) return true;
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

// One block computes the logits of kRouteTok tokens against all E experts, then one warp
// per token selects the top-k with warp shuffles and writes idx, w and the counts.
template <typename T>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const T* __restrict__ x, const T* __restrict__ Wg, const float* __restrict__ bg,
             int Tn, int d, int E, int k, float inv_temp, float noise_std, uint32_t noise_seed,
             int32_t* __restrict__ idx, float* __restrict__ w, int32_t* __restrict__ counts,
             float* __restrict__ logits) {
    pdl_wait();
    extern __shared__ float smem[];
    float* xs = smem;                                    // [kRouteTok][kRouteKc+1]
    float* wsm = xs + kRouteTok * (kRouteKc + 1);        // [E][kRouteKc+1]
    float* lg = wsm + E * (kRouteKc + 1);                // [kRouteTok][E]

    const int tid = threadIdx.x;
    const int tx = tid & 31, ty = tid >> 5;
    const int tok0 = blockIdx.x * kRouteTok;
    const int nb = (E + 31) / 32;                        // experts per lane (<= 8)

    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;

    for (int c0 = 0; c0 < d; c0 += kRouteKc) {
        for (int i = tid; i < kRouteTok * kRouteKc; i += kRouteThreads) {
            const int t = i / kRouteKc, c = i % kRouteKc;
            const int tok = tok0 + t, col = c0 + c;
            xs[t * (kRouteKc + 1) + c] = (tok < Tn && col < d) ? ld_f(x + (size_t)tok * d + col) : 0.f;
        }
        for (int i = tid; i < E * kRouteKc; i += kRouteThreads) {
            const int e = i / kRouteKc, c = i % kRouteKc;
            const int col = c0 + c;
            wsm[e * (kRouteKc + 1) + c] = (col < d) ? ld_f(Wg + (size_t)e * d + col) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < kRouteKc; ++c) {
            float xv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) xv[a] = xs[(ty + 8 * a) * (kRouteKc + 1) + c];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (b < nb) {
                    const int e = tx + 32 * b;
                    const float wv = (e < E) ? wsm[e * (kRouteKc + 1) + c] : 0.f;
#pragma unroll
                    for (int a = 0; a < 4; ++a) acc[a][b] = fmaf(xv[a], wv, acc[a][b]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int e = tx + 32 * b;
            if (b < nb && e < E) {
                float v = acc[a][b] + (bg ? bg[e] : 0.f);
                if (noise_std > 0.f) v = fmaf(noise_std, routing_noise(tok0 + ty + 8 * a, e, noise_seed), v);
                lg[(ty + 8 * a) * E + e] = v;
                if (logits && tok0 + ty + 8 * a < Tn) logits[(size_t)(tok0 + ty + 8 * a) * E + e] = v;
            }
        }
    __syncthreads();

    if (k == E) {
        // dense soft routing: w[t, e] = softmax(z_t / temp)_e over all E, slot e = expert e
        for (int a = 0; a < 4; ++a) {
            const int t = ty + 8 * a;
            const int tok = tok0 + t;
            if (tok >= Tn) break;
            float m = -INFINITY;
            for (int e = tx; e < E; e += 32) m = fmaxf(m, lg[t * E + e]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float s = 0.f;
            for (int e = tx; e < E; e += 32) s += expf((lg[t * E + e] - m) * inv_temp);
            s = warp_sum(s);
            const float inv = 1.f / s;
            for (int e = tx; e < E; e += 32) {
                idx[(size_t)tok * E + e] = e;
                w[(size_t)tok * E + e] = expf((lg[t * E + e] - m) * inv_temp) * inv;
            }
        }
        return;
    }

    // top-k per token: warp ty handles tokens ty, ty+8, ty+16, ty+24
    for (int a = 0; a < 4; ++a) {
        const int t = ty + 8 * a;
        const int tok = tok0 + t;
        if (tok >= Tn) break;
        float v[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int e = tx + 32 * b;
            v[b] = (b < nb && e < E) ? lg[t * E + e] : -INFINITY;
        }
        float sel_v[MOE_MAX_K];
        int sel_e[MOE_MAX_K];
        unsigned taken = 0u;  // bit b: expert tx + 32*b already selected
        for (int j = 0; j < k; ++j) {
            // lane-local best (largest value, lowest id among equals)
            float bv = -INFINITY;
            int be = kNoExpert;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int e = tx + 32 * b;
                if (b < nb && e < E && !((taken >> b) & 1u) && beats(v[b], e, bv, be)) { bv = v[b]; be = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (beats(ov, oe, bv, be)) { bv = ov; be = oe; }
            }
            sel_v[j] = bv;
            sel_e[j] = be;
            if ((be & 31) == tx) taken |= 1u << (be >> 5);
        }
        if (tx == 0) {
            // softmax over the k selected values divided by the temperature
            const float m = sel_v[0];
            float p[MOE_MAX_K], s = 0.f;
            for (int j = 0; j < k; ++j) { p[j] = expf((sel_v[j] - m) * inv_temp); s += p[j]; }
            const float inv = 1.f / s;
            for (int j = 0; j < k; ++j) {
                idx[(size_t)tok * k + j] = sel_e[j];
                w[(size_t)tok * k + j] = p[j] * inv;
                atomicAdd(counts + sel_e[j], 1);
            }
        }
    }
}

// noise[e, t] = N(0,1) normal of (token t, expert e), expert-major so that the router's
// lanes (consecutive tokens) read consecutive addresses. One thread per (token, group of four
// experts): groups run over grid.y and tokens over grid.x.
__global__ void __launch_bounds__(256)
noise_kernel(int Tn, int E, uint32_t seed, float* __restrict__ noise) {
    pdl_wait();
    const int groups = (E + 3) >> 2;
    for (int g = blockIdx.y; g < groups; g += gridDim.y) {
        for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < Tn; t += gridDim.x * blockDim.x) {
            float z[4];
            routing_noise4(t, g, seed, z);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * g + j < E) noise[(size_t)(4 * g + j) * Tn + t] = z[j];
        }
    }
}

// balance_loss = mean over experts of (counts[e] - T*k/E)^2 (fp32: one warp, lanes over
// experts, a fixed-order butterfly; GB300's FP64 rate is far too low for a serial loop). With
// dense routing (dense_T >= 0) every expert's count is first set to dense_T, the token count.
__global__ void __launch_bounds__(32)
balance_loss_kernel(int32_t* __restrict__ counts, int E, float mean, int dense_T, float* __restrict__ out) {
    pdl_wait();
    const int lane = threadIdx.x;
    float s = 0.f;
    for (int e = lane; e < E; e += 32) {
        if (dense_T >= 0) counts[e] = dense_T;
        const float dv = (float)(dense_T >= 0 ? dense_T : counts[e]) - mean;
        s = fmaf(dv, dv, s);
    }
    s = warp_sum(s);
    if (lane == 0) *out = s / (float)E;
}

}  // namespace

cudaError_t launch_route(const moe_config_t& c, const void* x, const void* Wg, const float* bg,
                         int32_t* idx, float* w, int32_t* counts, float* balance_loss, float* logits,
                         float* noise, cudaStream_t s) {
    cudaError_t st = launch_fill(counts, (long long)c.E, (int32_t)0, s);
    if (st != cudaSuccess) return st;
    if (c.T > 0 && tc_route_supported(c)) {
        const bool noisy = c.noise_std > 0.f;
        if (noisy) {
            if (!noise) return cudaErrorInvalidValue;
            // one block row per group of four experts (E <= 256), about 16 blocks of 256 threads
            // per SM in all
            const int groups = (c.E + 3) / 4;
            const int gx = std::min(ceil_div(c.T, 256), std::max(1, num_sms() * 16 / groups));
            const dim3 grid((unsigned)gx, (unsigned)groups);
            st = launch_pdl(noise_kernel, grid, dim3(256), 0, s, c.T, c.E, c.noise_seed, noise);
            count_launch();
            if (st != cudaSuccess) return st;
        }
        st = launch_route_tc(c, x, Wg, bg, idx, w, counts, logits, noisy ? noise : nullptr, s);
        if (st != cudaSuccess) return st;
    } else if (c.T > 0) {
        const size_t smem = sizeof(float) * ((size_t)kRouteTok * (kRouteKc + 1) +
                                             (size_t)c.E * (kRouteKc + 1) + (size_t)kRouteTok * c.E);
        const int grid = ceil_div(c.T, kRouteTok);
        const float inv_temp = 1.0f / c.temperature;
        const float* bias = c.has_gate_bias ? bg : nullptr;
        if (c.dtype == MOE_BF16) {
            auto kern = route_kernel<__nv_bfloat16>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            launch_pdl(kern, grid, kRouteThreads, smem, s, (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wg,
                                                   bias, c.T, c.d, c.E, c.k, inv_temp, c.noise_std, c.noise_seed,
                                                   idx, w, counts, logits);
        } else {
            auto kern = route_kernel<float>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            launch_pdl(kern, grid, kRouteThreads, smem, s, (const float*)x, (const float*)Wg, bias, c.T, c.d,
                                                   c.E, c.k, inv_temp, c.noise_std, c.noise_seed, idx, w,
                                                   counts, logits);
        }
        count_launch();
        st = cudaGetLastError();
        if (st != cudaSuccess) return st;
    }
    const float mean = (float)((double)c.T * (double)c.k / (double)c.E);
    launch_pdl(balance_loss_kernel, 1, 32, 0, s, counts, c.E, mean, dense_routing(c) ? c.T : -1, balance_loss);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
