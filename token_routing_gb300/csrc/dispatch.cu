// Dispatch: expert histogram, exclusive scans, capacity drops, stable ranks, and the gather
// of token rows into expert buckets.
//
// "Native MoE training system PithTrain", section 4.3 item 1 (capacity = capacity_factor *
// tokens / num_experts; overflow tokens are dropped), and "Expert Parallelism: Scaling
// Mixture-of-Experts Models", section 4.2 idea 2 (each routed token is written straight to
// its expert bucket's offset instead of being concatenated).
//
// The sort is deterministic: the rank of assignment (t, j) -> e is the number of earlier
// tokens that picked e, computed as (per-chunk histogram -> column scan over chunks) +
// (population count of e's token bitmask inside the chunk). Buckets are padded to the row
// alignment (128 rows) so that every GEMM row tile belongs to exactly one expert.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kSortTok = 256;   // tokens per chunk (one block per chunk in both sort kernels)

// The sort in two launches, one block per chunk of kSortTok tokens:
//   sort_hist_kernel  the chunk's expert histogram (ids checked for range and repeats)
//   sort_rank_kernel  every block reads all chunk histograms: the expert totals (counts) and
//                     the sum over the chunks before its own (its rank base); then kept /
//                     bucket offsets / assignment offsets from the counts, and the ranks of its
//                     chunk's assignments from per-expert token bitmasks (population counts). It
//                     writes slot_row, row_token (padding rows -1) and the expert-major
//                     assignment list.
// The kernel boundary orders the two phases: there is no grid barrier and no co-residency
// requirement.
struct SortArgs {
    const int32_t* idx;
    int T, k, E, C, align, nchunk;
    int32_t* blk_hist;
    int32_t* assign_off;
    int32_t* assign_tok;
    int32_t* kept;       // bucket outputs: null in assignment-only mode
    int32_t* offsets;
    int32_t* row_token;
    int32_t* slot_row;
    int32_t* n_dropped;
    int* err;
};

// Exclusive scans of two arrays of n <= blockDim.x values in shared memory (blockDim.x a
// multiple of 32, at most 1024): warp scans by shuffles, then the warp totals. The totals are
// returned in *tot_a, *tot_b.
__device__ void block_exclusive_scan2(int* a, int* b, int n, int* tot_a, int* tot_b) {
    __shared__ int s_wa[32], s_wb[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int va = tid < n ? a[tid] : 0, vb = tid < n ? b[tid] : 0;
    int ia = va, ib = vb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, ia, off), xb = __shfl_up_sync(0xffffffffu, ib, off);
        if (lane >= off) { ia += xa; ib += xb; }
    }
    if (lane == 31) { s_wa[warp] = ia; s_wb[warp] = ib; }
    __syncthreads();
    int pa = 0, pb = 0, ta = 0, tb = 0;
    const int nw = (int)blockDim.x >> 5;
    for (int w = 0; w < nw; ++w) {
        if (w < warp) { pa += s_wa[w]; pb += s_wb[w]; }
        ta += s_wa[w]; tb += s_wb[w];
    }
    if (tid < n) { a[tid] = pa + ia - va; b[tid] = pb + ib - vb; }
    *tot_a = ta;
    *tot_b = tb;
    __syncthreads();
}

// The experts of token t's k slots, in slot order; -1 for an id out of range or repeated
// (reported through the error word when `report`).
__device__ __forceinline__ void token_experts(const SortArgs& a, int t, int (&mine)[MOE_MAX_K], bool report) {
    int id[MOE_MAX_K];
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) id[j] = j < a.k ? a.idx[(size_t)t * a.k + j] : -1;   // all loads in flight
#pragma unroll
    for (int j = 0; j < MOE_MAX_K; ++j) {
        mine[j] = -1;
        if (j >= a.k) continue;
        const int e = id[j];
        bool ok = (e >= 0 && e < a.E);
#pragma unroll
        for (int i = 0; i < j; ++i) ok = ok && (mine[i] != e);
        if (ok) mine[j] = e;
        else if (report) raise_error(a.err, kErrBounds);
    }
}

__global__ void __launch_bounds__(kSortTok)
sort_hist_kernel(SortArgs a) {
    __shared__ int s_h[MOE_MAX_EXPERTS];
    const int tid = threadIdx.x, ch = blockIdx.x;
    for (int e = tid; e < a.E; e += blockDim.x) s_h[e] = 0;
    pdl_wait();
    __syncthreads();
    const int t = ch * kSortTok + tid;
    if (t < a.T) {
        int mine[MOE_MAX_K];
        token_experts(a, t, mine, true);
        for (int j = 0; j < a.k; ++j)
            if (mine[j] >= 0) atomicAdd(&s_h[mine[j]], 1);
    }
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x) a.blk_hist[(size_t)ch * a.E + e] = s_h[e];
}

__global__ void __launch_bounds__(kSortTok)
sort_rank_kernel(SortArgs a) {
    constexpr int W = kSortTok / 32;      // mask words per expert
    __shared__ uint32_t s_mask[MOE_MAX_EXPERTS * W];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_aoff[MOE_MAX_EXPERTS + 1];
    __shared__ int s_kept[MOE_MAX_EXPERTS];
    __shared__ int s_cnt[MOE_MAX_EXPERTS];
    __shared__ int s_base[MOE_MAX_EXPERTS];
    __shared__ int s_part[2][kSortTok];
    const int tid = threadIdx.x;
    const int ch = blockIdx.x;
    const int t = ch * kSortTok + tid;
    const int word = tid >> 5;
    const uint32_t bit = 1u << (tid & 31);
    for (int i = tid; i < a.E * W; i += blockDim.x) s_mask[i] = 0u;
    pdl_wait();
    // this chunk's token bitmasks per expert (idx was checked by the histogram kernel)
    int mine[MOE_MAX_K];
    __syncthreads();
    if (t < a.T) {
        token_experts(a, t, mine, false);
        for (int j = 0; j < a.k; ++j)
            if (mine[j] >= 0) atomicOr(&s_mask[mine[j] * W + word], bit);
    } else {
#pragma unroll
        for (int j = 0; j < MOE_MAX_K; ++j) mine[j] = -1;
    }

    // expert totals and this chunk's prefix, from all chunk histograms: thread (g, e) sums
    // column e over the chunks c = g mod groups (consecutive threads read consecutive experts
    // of a chunk's row; many rows in flight per thread), then the group partials are added
    const int groups = max(1, kSortTok / a.E);
    {
        int tot = 0, pre = 0;
        if (tid < groups * a.E) {
            const int e = tid % a.E, g = tid / a.E;
            constexpr int R = 16;   // rows in flight per thread
            for (int c0 = g; c0 < a.nchunk; c0 += R * groups) {
                int v[R];
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const int c = c0 + i * groups;
                    v[i] = c < a.nchunk ? __ldcg(a.blk_hist + (size_t)c * a.E + e) : 0;
                }
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    tot += v[i];
                    pre += c0 + i * groups < ch ? v[i] : 0;
                }
            }
        }
        s_part[0][tid] = tot;
        s_part[1][tid] = pre;
    }
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x) {
        int tot = 0, pre = 0;
        for (int g = 0; g < groups; ++g) { tot += s_part[0][g * a.E + e]; pre += s_part[1][g * a.E + e]; }
        s_cnt[e] = tot;
        s_base[e] = pre;
    }
    __syncthreads();

    // offsets (every block computes them), then this chunk's ranks and the bucket layout
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int cnt = s_cnt[e];
        const int kept = min(cnt, a.C);
        s_kept[e] = kept;
        s_off[e] = (kept + a.align - 1) / a.align * a.align;
        s_aoff[e] = cnt;
    }
    __syncthreads();
    int rows_total, assign_total;
    block_exclusive_scan2(s_off, s_aoff, a.E, &rows_total, &assign_total);
    if (tid == 0) { s_off[a.E] = rows_total; s_aoff[a.E] = assign_total; }
    __syncthreads();
    if (ch == 0) {
        for (int e = tid; e <= a.E; e += blockDim.x) {
            a.assign_off[e] = s_aoff[e];
            if (a.offsets) a.offsets[e] = s_off[e];
            if (a.kept && e < a.E) a.kept[e] = s_kept[e];
        }
        if (a.n_dropped && tid == 0) {
            int tk = 0;
            for (int e = 0; e < a.E; ++e) tk += s_kept[e];
            *a.n_dropped = a.T * a.k - tk;
        }
    }
    // padding rows of the buckets this block owns
    if (a.row_token) {
        for (int e = ch; e < a.E; e += gridDim.x)
            for (int r = s_off[e] + s_kept[e] + tid; r < s_off[e + 1]; r += blockDim.x) a.row_token[r] = -1;
    }
    if (t < a.T) {
        for (int j = 0; j < a.k; ++j) {
            const int e = mine[j];
            if (e < 0) {
                if (a.slot_row) a.slot_row[(size_t)t * a.k + j] = -1;
                continue;
            }
            const uint32_t* m = s_mask + e * W;
            int local = __popc(m[word] & (bit - 1u));
            for (int w2 = 0; w2 < word; ++w2) local += __popc(m[w2]);
            const int rank = s_base[e] + local;
            a.assign_tok[s_aoff[e] + rank] = t * a.k + j;
            if (a.slot_row) {
                if (rank < a.C) {
                    const int row = s_off[e] + rank;
                    a.slot_row[(size_t)t * a.k + j] = row;
                    a.row_token[row] = t;
                } else {
                    a.slot_row[(size_t)t * a.k + j] = -1;
                }
            }
        }
    }
}

// Dense soft routing (k = E): every expert receives every token, so the sort has a closed
// form. kept = min(T, C); bucket e starts at e * B with B = kept rounded up to the alignment;
// slot (t, j) sits at row j * B + t when t < kept, else it is dropped. One thread per
// (token, slot) for slot_row (checking idx[t, j] = j) and per bucket row for row_token.
__global__ void __launch_bounds__(256)
dense_layout_kernel(const int32_t* __restrict__ idx, int T, int E, int C, int align, int32_t* __restrict__ kept,
                    int32_t* __restrict__ offsets, int32_t* __restrict__ row_token, int32_t* __restrict__ slot_row,
                    int32_t* __restrict__ n_dropped, int* err) {
    pdl_wait();
    const int kp = min(T, C);
    const long long B = ((long long)kp + align - 1) / align * align;
    const long long n_slot = (long long)T * E;
    const long long n_rows = B * E;
    const long long stride = (long long)gridDim.x * blockDim.x;
    if (n_slot + n_rows + stride <= 0x7fffffffLL) {
        // 32-bit index arithmetic (a 64-bit division per item is a long software sequence)
        const int ns = (int)n_slot, nt = (int)(n_slot + n_rows), b = (int)B;
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nt; i += (int)stride) {
            if (i < ns) {
                const int t = i / E, j = i - t * E;
                const bool ok = idx[i] == j;
                if (!ok) raise_error(err, kErrBounds);
                slot_row[i] = (ok && t < kp) ? j * b + t : -1;
            } else {
                const int r = i - ns;
                const int rr = r % b;
                row_token[r] = rr < kp ? rr : -1;
            }
        }
    } else {
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_slot + n_rows; i += stride) {
            if (i < n_slot) {
                const int t = (int)(i / E), j = (int)(i % E);
                const bool ok = idx[i] == j;
                if (!ok) raise_error(err, kErrBounds);
                slot_row[i] = (ok && t < kp) ? (int32_t)(j * B + t) : -1;
            } else {
                const long long r = i - n_slot;
                const int rr = (int)(r % B);
                row_token[r] = rr < kp ? rr : -1;
            }
        }
    }
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            offsets[e] = (int32_t)(e * B);
            if (e < E) kept[e] = kp;
        }
        if (threadIdx.x == 0) *n_dropped = (T - kp) * E;
    }
}

// Xp[slot_row[t, j]] = x[t] for every kept slot, one warp per token (x read once, stored to
// each of its rows; slots in groups of G); then the padding rows (row_token = -1) below
// offsets[E] are zeroed, 32 rows per warp at a time (ballot, then coalesced stores).
template <typename T, int G>
__global__ void __launch_bounds__(256)
gather_kernel(const T* __restrict__ x, const int32_t* __restrict__ offsets, int E,
              const int32_t* __restrict__ row_token, const int32_t* __restrict__ slot_row, int Tn, int k,
              int d, int rows_cap, T* __restrict__ Xp) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    for (int t = gw; t < Tn; t += nwarps) {
        for (int j0 = 0; j0 < k; j0 += G) {
            int rows[G];
#pragma unroll
            for (int j = 0; j < G; ++j) rows[j] = j0 + j < k ? slot_row[(size_t)t * k + j0 + j] : -1;
            if ((d % V) == 0) {
                for (int c = lane * V; c < d; c += 32 * V) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + c));
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (rows[j] >= 0) *reinterpret_cast<uint4*>(Xp + (size_t)rows[j] * d + c) = v;
                }
            } else {
                for (int c = lane; c < d; c += 32) {
                    const T v = x[(size_t)t * d + c];
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (rows[j] >= 0) Xp[(size_t)rows[j] * d + c] = v;
                }
            }
        }
    }
    const int nrows = min(offsets[E], rows_cap);
    for (int r0 = gw * 32; r0 < nrows; r0 += nwarps * 32) {
        const int r = r0 + lane;
        unsigned pad = __ballot_sync(0xffffffffu, r < nrows && row_token[r] < 0);
        while (pad) {
            const int b = __ffs(pad) - 1;
            pad &= pad - 1;
            T* out = Xp + (size_t)(r0 + b) * d;
            if ((d % V) == 0) {
                for (int c = lane * V; c < d; c += 32 * V) *reinterpret_cast<uint4*>(out + c) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                for (int c = lane; c < d; c += 32) out[c] = Elem<T>::from_f(0.f);
            }
        }
    }
}

// Rows of each bucket that hold an assignment. They come first in the bucket, and the
// padding after them (row_token -1) is shorter than the row alignment, so the first padding
// row is found by a binary search over the bucket's last align - 1 rows.
__global__ void __launch_bounds__(256)
bucket_used_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_token, int E, int align,
                   int32_t* __restrict__ used) {
    pdl_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int lo = offsets[e], hi = offsets[e + 1];
    int a = max(lo, hi - (align - 1)), b = hi;   // the first padding row is in [a, b] (b: none)
    while (a < b) {
        const int m = (a + b) >> 1;
        if (row_token[m] < 0) b = m;
        else a = m + 1;
    }
    used[e] = a - lo;
}

}  // namespace

cudaError_t launch_bucket_used(const moe_config_t& c, const int32_t* offsets, const int32_t* row_token,
                               int32_t* used, cudaStream_t st) {
    if (c.E <= 0) return cudaSuccess;
    cudaError_t e = launch_pdl(bucket_used_kernel, ceil_div(c.E, 256), 256, 0, st, offsets, row_token, c.E,
                               c.row_align, used);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int sort_blocks(int T) { return T > 0 ? ceil_div(T, kSortTok) : 1; }

void sort_scratch_take(Workspace& ws, const moe_config_t& c, SortScratch* s) {
    const int nblk = sort_blocks(c.T);
    s->blk_hist = ws.take<int32_t>((size_t)nblk * c.E);
    s->assign_off = ws.take<int32_t>((size_t)c.E + 1);
    s->assign_tok = ws.take<int32_t>((size_t)c.T * c.k + 1);
}

cudaError_t launch_sort(const moe_config_t& c, const int32_t* idx, const SortScratch& s,
                        int32_t* kept, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                        int32_t* n_dropped, cudaStream_t st) {
    SortArgs a{};
    a.idx = idx; a.T = c.T; a.k = c.k; a.E = c.E; a.C = c.capacity; a.align = c.row_align;
    a.nchunk = sort_blocks(c.T);
    a.blk_hist = s.blk_hist;
    a.assign_off = s.assign_off; a.assign_tok = s.assign_tok;
    a.kept = kept; a.offsets = offsets; a.row_token = row_token; a.slot_row = slot_row;
    a.n_dropped = n_dropped; a.err = device_error_word();
    cudaError_t e = launch_pdl(sort_hist_kernel, a.nchunk, kSortTok, 0, st, a);
    count_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(sort_rank_kernel, a.nchunk, kSortTok, 0, st, a);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_dense_layout(const moe_config_t& c, const int32_t* idx, int32_t* kept, int32_t* offsets,
                                int32_t* row_token, int32_t* slot_row, int32_t* n_dropped, cudaStream_t st) {
    const long long items = (long long)c.T * c.E + (long long)c.rows_capacity;
    const int grid = (int)std::max(1LL, std::min((items + 255) / 256, (long long)num_sms() * 8));
    launch_pdl(dense_layout_kernel, grid, 256, 0, st, idx, c.T, c.E, c.capacity, c.row_align, kept, offsets, row_token,
                                              slot_row, n_dropped, device_error_word());
    count_launch();
    return cudaGetLastError();
}

template <typename T, int G>
static cudaError_t gather_g(const moe_config_t& c, const void* x, const int32_t* offsets, const int32_t* row_token,
                            const int32_t* slot_row, void* Xp, cudaStream_t st) {
    const long long warps = std::max<long long>(c.T, 1);
    const int grid = (int)std::max(1LL, std::min((warps + 7) / 8, (long long)num_sms() * 16));
    return launch_pdl(gather_kernel<T, G>, grid, 256, 0, st, (const T*)x, offsets, c.E, row_token, slot_row, c.T,
                      c.k, c.d, c.rows_capacity, (T*)Xp);
}
template <typename T>
static cudaError_t gather_t(const moe_config_t& c, const void* x, const int32_t* offsets, const int32_t* row_token,
                            const int32_t* slot_row, void* Xp, cudaStream_t st) {
    if (c.k <= 1) return gather_g<T, 1>(c, x, offsets, row_token, slot_row, Xp, st);
    if (c.k <= 2) return gather_g<T, 2>(c, x, offsets, row_token, slot_row, Xp, st);
    if (c.k <= 4) return gather_g<T, 4>(c, x, offsets, row_token, slot_row, Xp, st);
    return gather_g<T, 8>(c, x, offsets, row_token, slot_row, Xp, st);
}

cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* offsets,
                          const int32_t* row_token, const int32_t* slot_row, void* Xp, cudaStream_t st) {
    if (c.rows_capacity == 0) return cudaSuccess;
    cudaError_t e = c.dtype == MOE_BF16 ? gather_t<__nv_bfloat16>(c, x, offsets, row_token, slot_row, Xp, st)
                                        : gather_t<float>(c, x, offsets, row_token, slot_row, Xp, st);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
