// Dispatch: expert histogram, exclusive scans, capacity drops, stable ranks, and the gather
// of token rows into expert buckets.
//
// "Native MoE training system PithTrain", section 4.3 item 1 (capacity = capacity_factor *
// tokens / num_experts; overflow tokens are dropped), and "Expert Parallelism: Scaling
// Mixture-of-Experts Models", section 4.2 idea 2 (each routed token is written straight to
// its expert bucket's offset instead of being concatenated).
//
// The sort is deterministic: the rank of assignment (t, j) -> e is the number of earlier
// tokens that picked e, computed as (per-block histogram -> column scan over blocks) +
// (ordered rank inside the block). Buckets are padded to the configured alignment (128 or
// 256 rows) so that every GEMM row tile belongs to exactly one expert.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kSortTok = 256;   // tokens per block in the histogram / rank kernels

__global__ void __launch_bounds__(kSortTok)
hist_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ blk_hist,
            int* err) {
    __shared__ int h[MOE_MAX_EXPERTS];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kSortTok + threadIdx.x;
    if (t < T) {
        int mine[MOE_MAX_K];
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            bool ok = (e >= 0 && e < E);
            for (int i = 0; i < j; ++i) ok = ok && (mine[i] != e);
            mine[j] = ok ? e : -1;
            if (ok) atomicAdd(&h[e], 1);
            else raise_error(err, kErrBounds);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) blk_hist[(size_t)blockIdx.x * E + e] = h[e];
}

// One block, thread e: column scan of the block histograms, counts, kept = min(counts, C),
// bucket offsets (exclusive scan of kept rounded up to the bucket alignment), assignment offsets
// (exclusive scan of counts), n_dropped.
__global__ void __launch_bounds__(MOE_MAX_EXPERTS)
scan_kernel(const int32_t* __restrict__ blk_hist, int nblk, int E, int T, int k, int C, int align,
            int32_t* __restrict__ blk_base, int32_t* __restrict__ counts_out,
            int32_t* __restrict__ assign_off, int32_t* __restrict__ kept_out,
            int32_t* __restrict__ offsets, int32_t* __restrict__ n_dropped) {
    __shared__ int s_pad[MOE_MAX_EXPERTS];
    __shared__ int s_cnt[MOE_MAX_EXPERTS];
    __shared__ int s_kept[MOE_MAX_EXPERTS];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int b = 0; b < nblk; ++b) {
            const int v = blk_hist[(size_t)b * E + e];
            blk_base[(size_t)b * E + e] = run;
            run += v;
        }
    }
    const int kept = (e < E) ? min(run, C) : 0;
    s_cnt[e] = (e < E) ? run : 0;
    s_kept[e] = kept;
    s_pad[e] = (kept + align - 1) / align * align;
    __syncthreads();
    if (e == 0) {
        // E <= 256 sequential prefix sums: exact and deterministic
        int off = 0, aoff = 0, total_kept = 0;
        for (int i = 0; i < E; ++i) {
            if (offsets) offsets[i] = off;
            assign_off[i] = aoff;
            off += s_pad[i];
            aoff += s_cnt[i];
            total_kept += s_kept[i];
        }
        if (offsets) offsets[E] = off;
        assign_off[E] = aoff;
        if (n_dropped) *n_dropped = T * k - total_kept;
    }
    if (e < E) {
        counts_out[e] = run;
        if (kept_out) kept_out[e] = kept;
    }
}

// Ranks inside a block, without any order-dependent step: every (token, slot) sets its
// token's bit in a per-expert 256-bit mask, then the rank of token t among the block's
// tokens that picked e is the population count of e's mask below bit t. Writes the
// expert-major assignment list and, when the bucket outputs are requested, slot_row and
// row_token.
__global__ void __launch_bounds__(kSortTok)
rank_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int C,
            const int32_t* __restrict__ blk_base, const int32_t* __restrict__ assign_off,
            const int32_t* __restrict__ offsets, int32_t* __restrict__ assign_tok,
            int32_t* __restrict__ slot_row, int32_t* __restrict__ row_token) {
    constexpr int W = kSortTok / 32;
    __shared__ uint32_t s_mask[MOE_MAX_EXPERTS * W];
    for (int i = threadIdx.x; i < E * W; i += blockDim.x) s_mask[i] = 0u;
    __syncthreads();
    const int t = blockIdx.x * kSortTok + threadIdx.x;
    const int word = threadIdx.x >> 5;
    const uint32_t bit = 1u << (threadIdx.x & 31);
    int mine[MOE_MAX_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) mine[j] = -1;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            bool ok = (e >= 0 && e < E);
            for (int i = 0; i < j; ++i) ok = ok && (mine[i] != e);  // repeats were rejected by the histogram
            if (ok) {
                mine[j] = e;
                atomicOr(&s_mask[e * W + word], bit);
            }
        }
    }
    __syncthreads();
    if (t >= T) return;
    for (int j = 0; j < k; ++j) {
        const int e = mine[j];
        if (e < 0) continue;
        const uint32_t* m = s_mask + e * W;
        int local = __popc(m[word] & (bit - 1u));
        for (int w2 = 0; w2 < word; ++w2) local += __popc(m[w2]);
        const int rank = blk_base[(size_t)blockIdx.x * E + e] + local;
        assign_tok[assign_off[e] + rank] = t * k + j;
        if (slot_row) {
            if (rank < C) {
                const int row = offsets[e] + rank;
                slot_row[(size_t)t * k + j] = row;
                row_token[row] = t;
            } else {
                slot_row[(size_t)t * k + j] = -1;
            }
        }
    }
}

// Xp[r] = x[row_token[r]] for r < offsets[E]; padding rows (row_token = -1) are zeroed.
// One warp per row, 16-byte vectors when the row length allows.
template <typename T>
__global__ void __launch_bounds__(256)
gather_kernel(const T* __restrict__ x, const int32_t* __restrict__ offsets, int E,
              const int32_t* __restrict__ row_token, int d, int rows_cap, T* __restrict__ Xp) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nrows = min(offsets[E], rows_cap);
    constexpr int V = Vec16<T>::N;
    for (int r = warp; r < nrows; r += (gridDim.x * blockDim.x) >> 5) {
        const int t = row_token[r];
        T* dst = Xp + (size_t)r * d;
        if ((d % V) == 0) {
            for (int c = lane * V; c < d; c += 32 * V) {
                float v[V];
                if (t >= 0) load16(x + (size_t)t * d + c, v);
                else {
#pragma unroll
                    for (int i = 0; i < V; ++i) v[i] = 0.f;
                }
                store16(dst + c, v);
            }
        } else {
            for (int c = lane; c < d; c += 32) st_f(dst + c, t >= 0 ? ld_f(x + (size_t)t * d + c) : 0.f);
        }
    }
}

}  // namespace

int sort_blocks(int T) { return T > 0 ? ceil_div(T, kSortTok) : 1; }

void sort_scratch_take(Workspace& ws, const moe_config_t& c, SortScratch* s) {
    const int nblk = sort_blocks(c.T);
    s->blk_hist = ws.take<int32_t>((size_t)nblk * c.E);
    s->blk_base = ws.take<int32_t>((size_t)nblk * c.E);
    s->assign_off = ws.take<int32_t>((size_t)c.E + 1);
    s->assign_tok = ws.take<int32_t>((size_t)c.T * c.k + 1);
    s->counts = ws.take<int32_t>((size_t)c.E);
}

cudaError_t launch_sort(const moe_config_t& c, const int32_t* idx, const SortScratch& s,
                        int32_t* kept, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                        int32_t* n_dropped, cudaStream_t st) {
    const int nblk = sort_blocks(c.T);
    int* err = device_error_word();
    if (c.T == 0) {
        cudaError_t e = cudaMemsetAsync(s.blk_hist, 0, sizeof(int32_t) * c.E, st);
        if (e != cudaSuccess) return e;
    } else {
        hist_kernel<<<nblk, kSortTok, 0, st>>>(idx, c.T, c.k, c.E, s.blk_hist, err);
        count_launch();
    }
    scan_kernel<<<1, MOE_MAX_EXPERTS, 0, st>>>(s.blk_hist, nblk, c.E, c.T, c.k, c.capacity, c.row_align,
                                               s.blk_base, s.counts, s.assign_off, kept, offsets,
                                               n_dropped);
    count_launch();
    if (row_token) {
        cudaError_t e = cudaMemsetAsync(row_token, 0xff, sizeof(int32_t) * (size_t)c.rows_capacity, st);
        if (e != cudaSuccess) return e;
    }
    if (slot_row && c.T > 0) {  // assignments rejected as invalid stay -1
        cudaError_t e = cudaMemsetAsync(slot_row, 0xff, sizeof(int32_t) * (size_t)c.T * c.k, st);
        if (e != cudaSuccess) return e;
    }
    if (c.T > 0) {
        rank_kernel<<<nblk, kSortTok, 0, st>>>(idx, c.T, c.k, c.E, c.capacity, s.blk_base,
                                               s.assign_off, offsets, s.assign_tok, slot_row,
                                               row_token);
        count_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* offsets,
                          const int32_t* row_token, void* Xp, cudaStream_t st) {
    if (c.rows_capacity == 0) return cudaSuccess;
    const int rows_per_block = 8;
    const int grid = ceil_div(c.rows_capacity, rows_per_block);
    if (c.dtype == MOE_BF16)
        gather_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)x, offsets, c.E,
                                                           row_token, c.d, c.rows_capacity,
                                                           (__nv_bfloat16*)Xp);
    else
        gather_kernel<float><<<grid, 256, 0, st>>>((const float*)x, offsets, c.E, row_token, c.d,
                                                   c.rows_capacity, (float*)Xp);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
