// Expert co-selection matrix of a batch ("Expert Parallelism: Scaling Mixture-of-Experts
// Models", section 3.2, step 1: how often two experts are chosen by the same token, the
// input of the page's affinity-aware placement).
//
// H[i][i] = tokens that chose i; for i != j, H[i][j] = tokens whose top-k holds i in an
// earlier slot (higher logit) than j, so that H + H^T is the symmetric co-occurrence count.
// Integer counts: the result does not depend on the order of the atomic additions.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kCoselThreads = 256;
constexpr int kCoselSmemE = 64;   // up to this many experts the block histogram lives in smem

// Tokens are handled one per thread; each adds its k diagonal and k(k-1)/2 ordered pairs.
template <bool SMEM>
__global__ void __launch_bounds__(kCoselThreads)
coselect_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ H, int* err) {
    pdl_wait();
    __shared__ int s_h[SMEM ? kCoselSmemE * kCoselSmemE : 1];
    if (SMEM) {
        for (int i = threadIdx.x; i < E * E; i += blockDim.x) s_h[i] = 0;
        __syncthreads();
    }
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        int sel[MOE_MAX_K];
        int n = 0;
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            bool ok = (e >= 0 && e < E);
            for (int i = 0; i < n; ++i) ok = ok && (sel[i] != e);
            if (!ok) { raise_error(err, kErrBounds); continue; }
            sel[n++] = e;
        }
        for (int a = 0; a < n; ++a) {
            for (int b = a; b < n; ++b) {
                const int cell = sel[a] * E + sel[b];   // b == a: the diagonal count
                if (SMEM) atomicAdd(&s_h[cell], 1);
                else atomicAdd(H + cell, 1);
            }
        }
    }
    if (SMEM) {
        __syncthreads();
        for (int i = threadIdx.x; i < E * E; i += blockDim.x)
            if (s_h[i]) atomicAdd(H + i, s_h[i]);
    }
}

// Dense routing (k = E, slot j = expert j): every valid token adds 1 to H[i][j] for all
// i <= j. Counts the tokens whose idx row is the identity (others set MOE_ERR_DEVICE_BOUNDS)
// into H[0][0]; coselect_dense_fill_kernel then copies the count to every cell i <= j.
__global__ void __launch_bounds__(kCoselThreads)
coselect_dense_count_kernel(const int32_t* __restrict__ idx, int T, int E, int32_t* __restrict__ H, int* err) {
    pdl_wait();
    __shared__ int s_n;
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    int n = 0;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        bool ok = true;
        for (int j = 0; j < E; ++j) ok = ok && idx[(size_t)t * E + j] == j;
        if (ok) ++n;
        else raise_error(err, kErrBounds);
    }
    if (n) atomicAdd(&s_n, n);
    __syncthreads();
    if (threadIdx.x == 0 && s_n) atomicAdd(H, s_n);
}

__global__ void __launch_bounds__(kCoselThreads)
coselect_dense_fill_kernel(int E, int32_t* __restrict__ H) {
    pdl_wait();
    const int32_t n = H[0];
    __syncthreads();
    for (int c = threadIdx.x; c < E * E; c += blockDim.x) {
        const int i = c / E, j = c % E;
        if (i <= j) H[c] = n;
    }
}

}  // namespace

cudaError_t launch_coselect(const moe_config_t& c, const int32_t* idx, int32_t* H, cudaStream_t s) {
    cudaError_t e = launch_fill(H, (long long)c.E * c.E, (int32_t)0, s);
    if (e != cudaSuccess || c.T == 0) return e;
    const int grid = std::max(1, std::min(ceil_div(c.T, kCoselThreads), 2 * num_sms()));
    if (dense_routing(c) && c.k > MOE_MAX_K) {
        launch_pdl(coselect_dense_count_kernel, grid, kCoselThreads, 0, s, idx, c.T, c.E, H, device_error_word());
        count_launch();
        launch_pdl(coselect_dense_fill_kernel, 1, kCoselThreads, 0, s, c.E, H);
        count_launch();
        return cudaGetLastError();
    }
    if (c.E <= kCoselSmemE)
        launch_pdl(coselect_kernel<true>, grid, kCoselThreads, 0, s, idx, c.T, c.k, c.E, H, device_error_word());
    else
        launch_pdl(coselect_kernel<false>, grid, kCoselThreads, 0, s, idx, c.T, c.k, c.E, H, device_error_word());
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
