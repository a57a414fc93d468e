// Grouped expert GEMMs on CUDA cores (fp32 FMA, fp32 accumulation). They serve the fp32
// layer, whose 1e-4 tolerance rules out TF32 tensor cores, and bf16 shapes the tcgen05
// kernel does not take (d or d_ff not a multiple of 64).
//
// The per-expert FFN is Linear(d, d_ff) -> GELU -> Linear(d_ff, d) with biases
// ("PyTorch distributed MoE training", section 3.2, Expert; "Native MoE training system
// PithTrain", section 4.1, expert_pool); the backward GEMMs are its transposes.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kThreads = 256;

__device__ __forceinline__ int expert_of_row(const int32_t* offsets, int E, int row) {
    // largest e with offsets[e] <= row (buckets are non-empty ranges or empty)
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// C[r, n] = sum_k A[r, k] * B_e(n, k) over 64x64 tiles of bucket rows; 4x4 outputs per thread.
template <typename T>
__global__ void __launch_bounds__(kThreads)
row_gemm_simt_kernel(RowGemmArgs a) {
    pdl_wait();
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Bs[kBK][kBN + 4];
    const int m0 = blockIdx.y * kBM;
    const int n0 = blockIdx.x * kBN;
    const int rows_used = min(a.offsets[a.E], a.rows_capacity);
    if (m0 >= rows_used) return;
    const int e = expert_of_row(a.offsets, a.E, m0);
    const T* A = static_cast<const T*>(a.A);
    const T* B = static_cast<const T*>(a.B) + (size_t)e * a.sBe;
    const int tid = threadIdx.x;
    const int tr = tid / 16, tc = tid % 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < a.K; k0 += kBK) {
        for (int i = tid; i < kBM * kBK; i += kThreads) {
            const int r = i / kBK, kk = i % kBK;
            const int gk = k0 + kk;
            As[kk][r] = (gk < a.K) ? ld_f(A + (size_t)(m0 + r) * a.K + gk) : 0.f;
        }
        for (int i = tid; i < kBN * kBK; i += kThreads) {
            // B is walked along its contiguous index
            int n, kk;
            if (a.sBk == 1) { n = i / kBK; kk = i % kBK; } else { kk = i / kBN; n = i % kBN; }
            const int gn = n0 + n, gk = k0 + kk;
            Bs[kk][n] = (gn < a.N && gk < a.K) ? ld_f(B + gn * a.sBn + gk * a.sBk) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = As[kk][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tc * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    T* out0 = static_cast<T*>(a.out0);
    T* out1 = static_cast<T*>(a.out1);
    const T* bias = static_cast<const T*>(a.bias);
    const T* aux = static_cast<const T*>(a.aux);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = m0 + tr * 4 + i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tc * 4 + j;
            if (n >= a.N) continue;
            const size_t o = (size_t)r * a.N + n;
            float v = acc[i][j];
            switch (a.kind) {
                case kGemmFfn1: {
                    v += ld_f(bias + (size_t)e * a.N + n);
                    st_f(out0 + o, gelu_grad_f(v));  // saved for the backward
                    st_f(out1 + o, gelu_f(v));
                    break;
                }
                case kGemmFfn2:
                    st_f(out0 + o, v + ld_f(bias + (size_t)e * a.N + n));
                    break;
                case kGemmDH:
                    st_f(out0 + o, v * ld_f(aux + o));
                    break;
                default:
                    st_f(out0 + o, v);
                    break;
            }
        }
    }
}

// C_e[m, n] = sum over rows r of bucket e of P[r, m] * Q[r, n].
template <typename T>
__global__ void __launch_bounds__(kThreads)
wgrad_simt_kernel(WgradArgs a) {
    pdl_wait();
    __shared__ float Ps[kBK][kBM + 4];
    __shared__ float Qs[kBK][kBN + 4];
    const int e = blockIdx.z;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
    const int r0 = a.offsets[e], r1 = a.offsets[e + 1];
    const T* P = static_cast<const T*>(a.P);
    const T* Q = static_cast<const T*>(a.Q);
    const int tid = threadIdx.x;
    const int tr = tid / 16, tc = tid % 16;
    float acc[4][4] = {};
    for (int k0 = r0; k0 < r1; k0 += kBK) {
        for (int i = tid; i < kBK * kBM; i += kThreads) {
            const int kk = i / kBM, m = i % kBM;
            const int gr = k0 + kk, gm = m0 + m;
            Ps[kk][m] = (gr < r1 && gm < a.M) ? ld_f(P + (size_t)gr * a.M + gm) : 0.f;
        }
        for (int i = tid; i < kBK * kBN; i += kThreads) {
            const int kk = i / kBN, n = i % kBN;
            const int gr = k0 + kk, gn = n0 + n;
            Qs[kk][n] = (gr < r1 && gn < a.N) ? ld_f(Q + (size_t)gr * a.N + gn) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float pv[4], qv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = Ps[kk][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) qv[j] = Qs[kk][tc * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(pv[i], qv[j], acc[i][j]);
        }
        __syncthreads();
    }
    T* C = static_cast<T*>(a.C) + (size_t)e * a.M * a.N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + tr * 4 + i;
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tc * 4 + j;
            if (n < a.N) st_f(C + (size_t)m * a.N + n, acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t launch_row_gemm_simt(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s) {
    if (a.rows_capacity == 0) return cudaSuccess;
    dim3 grid(ceil_div(a.N, kBN), ceil_div(a.rows_capacity, kBM));
    if (c.dtype == MOE_BF16) launch_pdl(row_gemm_simt_kernel<__nv_bfloat16>, grid, kThreads, 0, s, a);
    else launch_pdl(row_gemm_simt_kernel<float>, grid, kThreads, 0, s, a);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_wgrad_simt(const moe_config_t& c, const WgradArgs& a, cudaStream_t s) {
    dim3 grid(ceil_div(a.N, kBN), ceil_div(a.M, kBM), a.E);
    if (c.dtype == MOE_BF16) launch_pdl(wgrad_simt_kernel<__nv_bfloat16>, grid, kThreads, 0, s, a);
    else launch_pdl(wgrad_simt_kernel<float>, grid, kThreads, 0, s, a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
