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
#include "tc_gemm_common.cuh"

namespace moe {

namespace {

using namespace tc;

// ------------------------------------------------------------------------- the kernel
template <int KIND, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmO0,
               const __grid_constant__ CUtensorMap tmO1) {
    constexpr bool WGRAD = (KIND == kGemmWgrad);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stg_smem = smem + STAGES * STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(stg_smem + EPI_SMEM);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_fail = reinterpret_cast<volatile int*>(tmem_slot + 1);  // a role gave up
    int* s_off = reinterpret_cast<int*>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(tfull + b, 1); mbar_init(tempty + b, EPI_THREADS); }
        mbar_init(drain, 1);
        *s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmA); tma_prefetch_desc(&tmB); }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // everything above touches only this CTA's shared memory and TMEM, and overlaps the
    // previous kernel's tail; global memory is read from here on
    pdl_wait();
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = p.offsets[i];
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
                *s_fail = 1;
                // let every copy already issued land before shared memory goes away
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t j = first; j < it; ++j) mbar_wait(full + j % STAGES, (j / STAGES) & 1, p.err);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(A_MN, B_MN);
            // operand descriptors at stage 0, k = 0; a stage and a K step of UMMA_K advance the
            // start-address field (16-byte units) by constants (K-major: 32 bytes inside the
            // swizzle atom; MN-major: 16 rows)
            const uint32_t s0 = smem_u32(smem);
            const uint64_t a_desc0 = A_MN ? make_desc(s0, BK * 128, 1024) : make_desc(s0, 16, 1024);
            const uint64_t b_desc0 = B_MN ? make_desc(s0 + A_BYTES, BK * 128, 1024) : make_desc(s0 + A_BYTES, 16, 1024);
            constexpr uint32_t A_KSTEP = (A_MN ? UMMA_K * 128 : UMMA_K * 2) >> 4;
            constexpr uint32_t B_KSTEP = (B_MN ? UMMA_K * 128 : UMMA_K * 2) >> 4;
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
                    const uint64_t soff = (uint64_t)(s * (STAGE_BYTES >> 4));
                    const uint64_t ad = a_desc0 + soff, bd = b_desc0 + soff;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        tc_mma(d_tmem, ad + kk * A_KSTEP, bd + kk * B_KSTEP, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(empty + s);  // frees the stage once these MMAs have read it
                }
                if (!ok) break;
                tc_commit(tfull + buf);    // accumulator ready for the epilogue
            }
            if (!ok) *s_fail = 1;
            // drain: every MMA issued so far has completed before TMEM is released
            tc_commit(drain);
            mbar_wait(drain, 0, p.err);
        }
    } else {
        // ---------------- epilogue warps 2..9: TMEM lane quarter = warp % 4, column half
        const int quarter = warp & 3;
        const int c_lo = ((warp - 2) >> 2) * (BN / 2);
        Stager st{smem_u32(stg_smem + (warp - 2) * 2 * STG_BYTES), 0};
        uint32_t tl = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const Tile t = decode_tile<WGRAD>(p, s_off, tile);
            if (t.kblocks == 0) {
                // an expert with no rows: its weight-gradient tile is zero
                const int y = t.m0 + quarter * 32;
                const int cols = min(BN / 2, p.N - (t.n0 + c_lo));
                if (WGRAD && y < p.M && cols > 0)
                    st.store_zero(lane, st.acquire(lane), &tmO0, t.n0 + c_lo, (cols + 31) / 32, t.e * p.M + y);
                continue;
            }
            const int buf = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            ++tl;
            // side input of the first chunk, fetched while the accumulator is being produced:
            // the bias row (same for every lane) or, for dH, the saved GELU'(A) read coalesced
            // (lane l: row (l>>2)+8i of the warp's 32 rows, 16-byte segment l&3)
            const size_t aux_row0 = (size_t)(t.m0 + quarter * 32 + (lane >> 2));
            Raw32 next;
            if (t.n0 + c_lo < p.N) {
                if (has_bias<KIND>()) load_raw32(next, p.bias + (size_t)t.e * p.N + t.n0 + c_lo);
                if (KIND == kGemmDH)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        next.q[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + (aux_row0 + 8 * i) * p.N + t.n0 + c_lo + (lane & 3) * 8));
            }
            if (!mbar_wait(tfull + buf, aph, p.err)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN;
            // the heavy epilogues (Ffn1's GELU, dH's product with GELU') load the next
            // accumulator chunk from TMEM while processing the current one
            constexpr bool PREFETCH = KIND == kGemmFfn1 || KIND == kGemmDH;
            uint32_t acc[32];
            if (PREFETCH && t.n0 + c_lo < p.N) tmem_ld32(taddr + c_lo, acc);
            for (int c = c_lo; c < c_lo + BN / 2; c += 32) {
                if (t.n0 + c >= p.N) break;
                const int n = t.n0 + c;
                const Raw32 cur = next;
                const bool more = c + 32 < c_lo + BN / 2 && n + 32 < p.N;
                if (more && has_bias<KIND>()) load_raw32(next, p.bias + (size_t)t.e * p.N + n + 32);
                if (more && KIND == kGemmDH)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        next.q[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + (aux_row0 + 8 * i) * p.N + n + 32 + (lane & 3) * 8));
                if (!PREFETCH) tmem_ld32(taddr + c, acc);
                tmem_ld_wait_regs(acc);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
                if (PREFETCH && more) tmem_ld32(taddr + c + 32, acc);
                const int y = t.m0 + quarter * 32;
                if (KIND == kGemmWgrad) {
                    const uint32_t b = st.acquire(lane);
                    if (t.m0 + quarter * 32 < p.M) st.store(lane, b, v, &tmO0, n, t.e * p.M + y);
                } else if (KIND == kGemmFfn1 || KIND == kGemmFfn2) {
                    float bv[32];
                    unpack_raw32(cur, bv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] += bv[i];
                    if (KIND == kGemmFfn1) {
                        // H = GELU(A) for the second GEMM, GELU'(A) saved for the backward
                        float gp[32];
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            gelu_and_grad_f2(v[i], v[i + 1], v[i], v[i + 1], gp[i], gp[i + 1]);
                        uint32_t b = st.acquire(lane);
                        st.store(lane, b, gp, &tmO0, n, y);
                        b = st.acquire(lane);
                        st.store(lane, b, v, &tmO1, n, y);
                    } else {
                        const uint32_t b = st.acquire(lane);
                        st.store(lane, b, v, &tmO0, n, y);
                    }
                } else if (KIND == kGemmDH) {
                    // transpose the coalesced GELU'(A) chunk through the staging buffer: lane = row
                    const uint32_t b = st.acquire(lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i) sts128(sw64_addr(b, (lane >> 2) + 8 * i, lane & 3), cur.q[i]);
                    __syncwarp();
                    float a[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) unpack8(lds128(sw64_addr(b, lane, j)), a + 8 * j);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= a[i];  // a = GELU'(A) saved by the forward
                    st.store(lane, b, v, &tmO0, n, y);
                    if (p.colsum) {
                        // db1 partial of this tile's lane quarter (32 rows) from the staged dA chunk
                        const float2 cs = staged_colsum32(b, lane);
                        if (lane < 16)
                            *reinterpret_cast<float2*>(p.colsum + ((size_t)(t.m0 / BM) * 4 + quarter) * p.N + n +
                                                       2 * lane) = cs;
                    }
                } else {
                    const uint32_t b = st.acquire(lane);
                    st.store(lane, b, v, &tmO0, n, y);
                }
            }
            tc_fence_before();
            mbar_arrive(tempty + buf);
            if (*s_fail) break;
        }
        // every TMA store has finished before the CTA's shared memory is released
        if (lane == 0) bulk_wait_all();
        __syncwarp();
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

constexpr size_t kSmemBytes = 1024 /*align slack*/ + STAGES * STAGE_BYTES + EPI_SMEM + 16 * sizeof(uint64_t) +
                              16 + kMaxOffsets * sizeof(int);
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// ------------------------------------------------------------------------- host side
template <int KIND, bool A_MN, bool B_MN>
cudaError_t launch_kernel(const TcParams& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o0,
                          const CUtensorMap& o1, int grid, cudaStream_t s) {
    auto kern = tc_gemm_kernel<KIND, A_MN, B_MN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    launch_pdl(kern, grid, THREADS, kSmemBytes, s, p, a, b, o0, o1);
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
    p.colsum = a.colsum;
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
    // epilogue stores: 32 x 32 boxes, 64-byte swizzle (matches the staging layout)
    CUtensorMap to0, to1;
    if (!make_map_ex(&to0, a.out0, (uint64_t)a.N, (uint64_t)a.rows_capacity, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (a.kind == kGemmFfn1) {
        if (!make_map_ex(&to1, a.out1, (uint64_t)a.N, (uint64_t)a.rows_capacity, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        to1 = to0;
    }
    const long long max_tiles = (long long)p.m_tiles * p.n_tiles;
    const int grid = (int)std::max(1LL, std::min<long long>(max_tiles, num_sms()));
    switch (a.kind) {
        case kGemmFfn1: return launch_kernel<kGemmFfn1, false, false>(p, ta, tb, to0, to1, grid, s);
        case kGemmFfn2: return launch_kernel<kGemmFfn2, false, false>(p, ta, tb, to0, to1, grid, s);
        case kGemmDH: return launch_kernel<kGemmDH, false, true>(p, ta, tb, to0, to1, grid, s);
        case kGemmDX: return launch_kernel<kGemmDX, false, true>(p, ta, tb, to0, to1, grid, s);
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
    CUtensorMap to0;
    if (!make_map_ex(&to0, a.C, (uint64_t)a.N, (uint64_t)a.E * a.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    const long long tiles = (long long)a.E * p.m_tiles * p.n_tiles;
    const int grid = (int)std::max(1LL, std::min<long long>(tiles, num_sms()));
    return launch_kernel<kGemmWgrad, true, true>(p, ta, tb, to0, to0, grid, s);
}

}  // namespace moe
