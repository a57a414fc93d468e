// Grouped expert GEMMs on the 5th-generation tensor cores (sm_103a): tcgen05.mma with the
// fp32 accumulator in tensor memory (TMEM), operands staged in shared memory by TMA
// (cp.async.bulk.tensor, 128-byte swizzle), mbarrier pipelines, persistent CTAs.
//
// The expert FFN is Linear(d, d_ff) -> GELU -> Linear(d_ff, d) with biases ("PyTorch
// distributed MoE training", section 3.2, Expert; "Native MoE training system PithTrain",
// section 4.1, expert_pool), applied to each expert's bucket of routed tokens. The same
// kernel covers the forward GEMMs (GELU and bias fused in the epilogue) and the backward
// ones (dH with the GELU derivative fused, dX, and the weight gradients whose reduction runs
// over the bucket rows).
//
// CTA = 10 warps: warp 0 issues TMA loads, warp 1 owns TMEM and issues the MMAs (one
// thread), warps 2..9 drain the accumulator (tcgen05.ld) and run the epilogue (two warps
// per TMEM lane quarter, each on half of the tile's columns). The
// accumulator is double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile
// overlaps the MMAs of the next. Tiles are 128 x 256 x 64 (bf16, fp32 accumulate).
//
// Every wait is bounded: a wait that runs out records a device error, the roles unwind,
// in-flight copies and MMAs are drained, and TMEM is freed before the CTA exits.
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                    // one 128-byte swizzle atom of bf16 along K
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;         // two accumulator buffers
constexpr int EPI_WARPS = 8;                 // two per TMEM lane quarter, each on half the columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int kMaxOffsets = MOE_MAX_EXPERTS + 1;

struct TcParams {
    int kind;                 // GemmKind
    const int32_t* offsets;   // [E+1] bucket starts
    int E, N, K, M;           // row GEMMs: out [rows, N], K reduction; wgrad: C_e [M, N]
    int n_tiles, m_tiles;
    const __nv_bfloat16* bias;   // [E, N]
    const __nv_bfloat16* aux;    // [rows, N] (A of the forward, for dH)
    __nv_bfloat16* out0;
    __nv_bfloat16* out1;
    int* err;
};

// Instruction descriptor of kind::f16: bf16 x bf16 -> fp32, M = 128, N = BN.
__host__ __device__ constexpr uint32_t make_idesc(bool a_mn_major, bool b_mn_major) {
    return (1u << 4)                      // D format fp32
         | (1u << 7)                      // A format bf16
         | (1u << 10)                     // B format bf16
         | ((a_mn_major ? 1u : 0u) << 15) // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16) // B major-ness
         | ((uint32_t)(BN >> 3) << 17)    // N >> 3
         | ((uint32_t)(BM >> 4) << 24);   // M >> 4
}

// ------------------------------------------------------------------------- tile decode
struct Tile {
    int e, m0, n0, row0, kblocks;
};

__device__ __forceinline__ int bucket_of(const int* s_off, int E, int row) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <bool WGRAD>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, const int* s_off, int tile) {
    Tile t;
    const int nt = tile % p.n_tiles;
    const int rest = tile / p.n_tiles;
    t.n0 = nt * BN;
    if (WGRAD) {
        t.m0 = (rest % p.m_tiles) * BM;
        t.e = rest / p.m_tiles;
        t.row0 = s_off[t.e];
        t.kblocks = (s_off[t.e + 1] - s_off[t.e]) / BK;
    } else {
        t.m0 = rest * BM;
        t.e = bucket_of(s_off, p.E, t.m0);
        t.row0 = t.m0;
        t.kblocks = p.K / BK;
    }
    return t;
}

// ------------------------------------------------------------------------- epilogue
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) store16(dst + 8 * q, v + 8 * q);
}

template <int KIND>
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const Tile& t, int row_in_tile,
                                               int c, const uint32_t (&acc)[32], const float (&a)[32]) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
    const int n = t.n0 + c;
    if (KIND == kGemmWgrad) {
        const int m = t.m0 + row_in_tile;
        if (m < p.M) store_row32(p.out0 + ((size_t)t.e * p.M + m) * p.N + n, v);
        return;
    }
    const size_t o = (size_t)(t.m0 + row_in_tile) * p.N + n;
    if (KIND == kGemmFfn1 || KIND == kGemmFfn2) {
        const __nv_bfloat16* b = p.bias + (size_t)t.e * p.N + n;
        float bv[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) load16(b + 8 * q, bv + 8 * q);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bv[i];
        store_row32(p.out0 + o, v);
        if (KIND == kGemmFfn1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
            store_row32(p.out1 + o, v);
        }
    } else if (KIND == kGemmDH) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gelu_grad_f(a[i]);
        store_row32(p.out0 + o, v);
    } else {
        store_row32(p.out0 + o, v);
    }
}

template <int KIND>
__device__ __forceinline__ void epilogue_zero(const TcParams& p, const Tile& t, int row_in_tile, int c_lo) {
    // an expert with no rows: its weight-gradient tile is zero
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0.f;
    const int m = t.m0 + row_in_tile;
    if (m >= p.M) return;
    for (int c = c_lo; c < c_lo + BN / 2; c += 32)
        if (t.n0 + c < p.N) store_row32(p.out0 + ((size_t)t.e * p.M + m) * p.N + t.n0 + c, z);
}

// ------------------------------------------------------------------------- the kernel
template <int KIND, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB) {
    constexpr bool WGRAD = (KIND == kGemmWgrad);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = p.offsets[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(tfull + b, 1); mbar_init(tempty + b, EPI_THREADS); }
        mbar_init(drain, 1);
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmA); tma_prefetch_desc(&tmB); }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = WGRAD ? p.E * p.m_tiles * p.n_tiles : (s_off[p.E] / BM) * p.n_tiles;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const Tile t = decode_tile<WGRAD>(p, s_off, tile);
                for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(empty + s, ph ^ 1, p.err)) { ok = false; break; }
                    const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    mbar_expect_tx(full + s, STAGE_BYTES);
                    const int k0 = kb * BK;
                    if (!A_MN) {
                        tma_load_2d(sa, &tmA, k0, t.row0, full + s);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d(sa + j * (BK * 128), &tmA, t.m0 + 64 * j, t.row0 + k0, full + s);
                    }
                    if (!B_MN) {
                        tma_load_2d(sb, &tmB, k0, t.e * p.N + t.n0, full + s);
                    } else if (WGRAD) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(sb + j * (BK * 128), &tmB, t.n0 + 64 * j, t.row0 + k0, full + s);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(sb + j * (BK * 128), &tmB, t.n0 + 64 * j, t.e * p.K + k0, full + s);
                    }
                }
            }
            if (!ok) {
                s_fail = 1;
                // let every copy already issued land before shared memory goes away
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j) mbar_wait(full + j % STAGES, (j / STAGES) & 1, p.err);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(A_MN, B_MN);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const Tile t = decode_tile<WGRAD>(p, s_off, tile);
                if (t.kblocks == 0) continue;
                const int buf = tl & 1;
                const uint32_t aph = (tl >> 1) & 1;
                ++tl;
                if (!mbar_wait(tempty + buf, aph ^ 1, p.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < t.kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(full + s, ph, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        // K-major: step 32 bytes inside the swizzle atom; MN-major: step 16 rows
                        const uint64_t ad = A_MN ? make_desc(sa + kk * UMMA_K * 128, BK * 128, 1024)
                                                 : make_desc(sa + kk * UMMA_K * 2, 16, 1024);
                        const uint64_t bd = B_MN ? make_desc(sb + kk * UMMA_K * 128, BK * 128, 1024)
                                                 : make_desc(sb + kk * UMMA_K * 2, 16, 1024);
                        tc_mma(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(empty + s);  // frees the stage once these MMAs have read it
                }
                if (!ok) break;
                tc_commit(tfull + buf);    // accumulator ready for the epilogue
            }
            if (!ok) s_fail = 1;
            // drain: every MMA issued so far has completed before TMEM is released
            tc_commit(drain);
            mbar_wait(drain, 0, p.err);
        }
    } else {
        // ---------------- epilogue warps 2..9: TMEM lane quarter = warp % 4, column half
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const int c_lo = ((warp - 2) >> 2) * (BN / 2);
        uint32_t tl = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const Tile t = decode_tile<WGRAD>(p, s_off, tile);
            if (t.kblocks == 0) {
                if (WGRAD) epilogue_zero<KIND>(p, t, row_in_tile, c_lo);
                continue;
            }
            const int buf = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            ++tl;
            if (!mbar_wait(tfull + buf, aph, p.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN;
            for (int c = c_lo; c < c_lo + BN / 2; c += 32) {
                if (t.n0 + c >= p.N) break;
                float a[32];
                if (KIND == kGemmDH) {
                    // forward pre-activation of this row's 32 columns, fetched before the
                    // accumulator so the two latencies overlap
                    const size_t o = (size_t)(t.m0 + row_in_tile) * p.N + t.n0 + c;
#pragma unroll
                    for (int q = 0; q < 4; ++q) load16(p.aux + o + 8 * q, a + 8 * q);
                }
                uint32_t acc[32];
                tmem_ld32(taddr + c, acc);
                tmem_ld_wait();
                epilogue_chunk<KIND>(p, t, row_in_tile, c, acc, a);
            }
            tc_fence_before();
            mbar_arrive(tempty + buf);
            if (s_fail) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

constexpr size_t kSmemBytes = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 16 * sizeof(uint64_t) +
                              16 + kMaxOffsets * sizeof(int);

// ------------------------------------------------------------------------- host side
template <int KIND, bool A_MN, bool B_MN>
cudaError_t launch_kernel(const TcParams& p, const CUtensorMap& a, const CUtensorMap& b, int grid,
                          cudaStream_t s) {
    auto kern = tc_gemm_kernel<KIND, A_MN, B_MN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, THREADS, kSmemBytes, s>>>(p, a, b);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

bool tc_gemm_supported(const moe_config_t& c) {
    // shape rule only: if the driver's tensor-map encoder is missing, the launch fails loudly
    return c.dtype == MOE_BF16 && c.d % 64 == 0 && c.d_ff % 64 == 0;
}

cudaError_t launch_row_gemm_tc(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s) {
    if (a.rows_capacity == 0) return cudaSuccess;
    TcParams p{};
    p.kind = a.kind;
    p.offsets = a.offsets;
    p.E = a.E; p.N = a.N; p.K = a.K; p.M = 0;
    p.n_tiles = ceil_div(a.N, BN);
    p.m_tiles = a.rows_capacity / BM;
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.aux = static_cast<const __nv_bfloat16*>(a.aux);
    p.out0 = static_cast<__nv_bfloat16*>(a.out0);
    p.out1 = static_cast<__nv_bfloat16*>(a.out1);
    p.err = device_error_word();
    CUtensorMap ta, tb;
    // A: activations [rows, K], K-major tiles of 128 rows
    if (!make_map(&ta, a.A, (uint64_t)a.K, (uint64_t)a.rows_capacity, BM)) return cudaErrorInvalidValue;
    const bool b_mn = (a.sBn == 1);
    if (!b_mn) {
        // B(n, k) = W[e*N + n][k]: K-major, [E*N, K]
        if (!make_map(&tb, a.B, (uint64_t)a.K, (uint64_t)a.E * a.N, BN)) return cudaErrorInvalidValue;
    } else {
        // B(n, k) = W[e*K + k][n]: N-major, [E*K, N], boxes of 64 n x 64 k
        if (!make_map(&tb, a.B, (uint64_t)a.N, (uint64_t)a.E * a.K, BK)) return cudaErrorInvalidValue;
    }
    const long long max_tiles = (long long)p.m_tiles * p.n_tiles;
    const int grid = (int)std::max(1LL, std::min<long long>(max_tiles, num_sms()));
    switch (a.kind) {
        case kGemmFfn1: return launch_kernel<kGemmFfn1, false, false>(p, ta, tb, grid, s);
        case kGemmFfn2: return launch_kernel<kGemmFfn2, false, false>(p, ta, tb, grid, s);
        case kGemmDH: return launch_kernel<kGemmDH, false, true>(p, ta, tb, grid, s);
        case kGemmDX: return launch_kernel<kGemmDX, false, true>(p, ta, tb, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wgrad_tc(const moe_config_t& c, const WgradArgs& a, cudaStream_t s) {
    TcParams p{};
    p.kind = kGemmWgrad;
    p.offsets = a.offsets;
    p.E = a.E; p.N = a.N; p.M = a.M; p.K = 0;
    p.n_tiles = ceil_div(a.N, BN);
    p.m_tiles = ceil_div(a.M, BM);
    p.out0 = static_cast<__nv_bfloat16*>(a.C);
    p.err = device_error_word();
    CUtensorMap ta, tb;
    const uint64_t rows = (uint64_t)std::max(c.rows_capacity, 1);
    // A(m, k=row) = P[row][m]: M-major, boxes of 64 m x 64 rows; B(n, k=row) = Q[row][n]
    if (!make_map(&ta, a.P, (uint64_t)a.M, rows, BK)) return cudaErrorInvalidValue;
    if (!make_map(&tb, a.Q, (uint64_t)a.N, rows, BK)) return cudaErrorInvalidValue;
    const long long tiles = (long long)a.E * p.m_tiles * p.n_tiles;
    const int grid = (int)std::max(1LL, std::min<long long>(tiles, num_sms()));
    return launch_kernel<kGemmWgrad, true, true>(p, ta, tb, grid, s);
}

}  // namespace moe
