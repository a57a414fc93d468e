// Grouped expert GEMMs on CTA pairs: tcgen05.mma.cta_group::2 over 256 x 256 x 64 tiles.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile: each CTA stages its own
// 128 rows of A and its half (128 columns) of B, so a stage is 32 KB instead of 48 KB and six
// stages fit where four fitted before (about 1.5x deeper lookahead per SM, half the B traffic).
// The leader CTA (cluster rank 0) issues the MMAs for the pair; the accumulator rows of each
// CTA land in its own TMEM, and each CTA drains and stores its own 128 rows.
//
// Synchronisation: both CTAs' TMA loads complete on the leader's "full" barrier (the leader
// expects the pair's bytes); the leader's commits arrive on both CTAs' "empty" and
// "accumulator full" barriers (multicast); both CTAs' epilogue threads arrive on the leader's
// "accumulator empty" barrier. Every wait is bounded and records a device error on expiry.
// Cluster barriers order the barrier initialisation before any remote access, and the end of
// all work in both CTAs before the pair releases its TMEM.
//
// The arithmetic per kind is the same as the one-CTA kernel (gemm_tc.cu): the expert FFN
// Linear(d, d_ff) -> GELU -> Linear(d_ff, d) ("PyTorch distributed MoE training", section 3.2)
// and its backward.
#include "tc_gemm_common.cuh"

namespace moe {

namespace {

constexpr int P_BM = 256;                           // pair tile rows (128 per CTA)
constexpr int P_HALF = 128;
constexpr int P_A_BYTES = P_HALF * BK * 2;          // 16 KB per CTA
constexpr int P_B_BYTES = P_HALF * BK * 2;          // 16 KB per CTA: half of B's 256 columns
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;

// 8 epilogue warps (two per TMEM lane quarter, 128 columns each) that fetch the next chunk's
// accumulator columns and side input ahead of use. Ffn1 writes two outputs per chunk (GELU'
// and H): each of its warps keeps two staging buffer pairs, and its ring has five 32 KB stages
// instead of six. (Twelve Ffn1 epilogue warps, three per quarter with one buffer pair each,
// measured the same; sixteen without the fetch-ahead measured slower.)
template <int KIND> constexpr int pair_epi_warps() { return 8; }
template <int KIND> constexpr int pair_threads() { return 64 + 32 * pair_epi_warps<KIND>(); }
template <int KIND> constexpr int pair_stages() { return KIND == kGemmFfn1 ? 5 : 6; }
// staging buffer pairs per Ffn1 epilogue warp
template <int KIND> constexpr int pair_ffn1_nb() { return pair_epi_warps<KIND>() > 8 ? 1 : 2; }
template <int KIND> constexpr int pair_epi_bytes() {
    return pair_epi_warps<KIND>() * (KIND == kGemmFfn1 ? 2 * pair_ffn1_nb<KIND>() : 2) * STG_BYTES;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t o;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(addr), "r"(rank));
    return o;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA tile load into this CTA's shared memory that completes on the leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                                 uint32_t mbar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(mbar_cluster)
        : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}
// Arrives on the barrier at this shared-memory offset in both CTAs of the pair once the
// leader's MMAs issued so far have completed.
__device__ __forceinline__ void commit_pair_both(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"((uint16_t)3) : "memory");
}
__device__ __forceinline__ void commit_pair_local(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

struct PairTile {
    int e, m0, n0, row0, kblocks;
    int end;      // row GEMMs: first row past the tile's bucket (a half at or past it is not stored)
};

// Row GEMMs: pair tile r of the launch is the (r - pairs_before(e))-th 256-row tile of bucket e,
// the largest e with pairs_before(e) <= r (s_q: the odd-bucket prefix).
template <bool WGRAD>
__device__ __forceinline__ PairTile decode_pair_tile(const TcParams& p, const int* s_off, const uint16_t* s_q,
                                                     int tile) {
    PairTile t;
    const int nt = tile % p.n_tiles;
    const int rest = tile / p.n_tiles;
    t.n0 = nt * BN;
    if (WGRAD) {
        t.m0 = (rest % p.m_tiles) * P_BM;
        t.e = rest / p.m_tiles;
        t.row0 = s_off[t.e];
        // the K loop stops at the last k-block that holds a row of the bucket with an
        // assignment: the rows after it are zero padding and add nothing
        t.kblocks = p.rows_used ? (int)s_q[t.e] : (s_off[t.e + 1] - s_off[t.e]) / BK;
        t.end = 0;
    } else {
        t.e = bucket_of_pair(s_off, s_q, p.E, rest);
        t.m0 = s_off[t.e] + (rest - pairs_before(s_off, s_q, t.e)) * P_BM;
        t.row0 = t.m0;
        t.kblocks = p.K / BK;
        t.end = s_off[t.e + 1];
    }
    return t;
}

template <int KIND, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads<KIND>(), 1)
tc_gemm_pair_kernel(const TcParams p, const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmO0,
                    const __grid_constant__ CUtensorMap tmO1) {
    constexpr bool WGRAD = (KIND == kGemmWgrad || KIND == kGemmWgradF32);
    constexpr bool AUX = (KIND == kGemmDH || KIND == kGemmAccum);   // side input read per chunk
    constexpr int P_STAGES = pair_stages<KIND>();
    constexpr int PE_THREADS = 32 * pair_epi_warps<KIND>();
    // accumulator columns per epilogue warp: the tile's 32-column chunks spread over the warps of
    // a lane quarter (4 + 4 with two warps, 3 + 3 + 2 with three)
    constexpr int WPQ = pair_epi_warps<KIND>() / 4;
    constexpr int CHUNKS = BN / 32;
    // the heavy epilogues (Ffn1's GELU, dH's product with GELU') load the next accumulator
    // chunk from TMEM while processing the current one
    constexpr bool PREFETCH = KIND == kGemmFfn1 || KIND == kGemmDH;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stg_smem = smem + P_STAGES * P_STAGE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(stg_smem + pair_epi_bytes<KIND>());
    uint64_t* empty = full + P_STAGES;
    uint64_t* tfull = empty + P_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* s_fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
    uint16_t* s_q = reinterpret_cast<uint16_t*>(s_off + kMaxOffsets);   // odd-bucket prefix (row GEMMs)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = (rank == 0);
    const int cluster_id = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(tfull + b, 1); mbar_init(tempty + b, 2 * PE_THREADS); }
        mbar_init(drain, 1);
        *s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmA); tma_prefetch_desc(&tmB); }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    // everything above touches only this CTA's shared memory and TMEM, and overlaps the
    // previous kernel's tail; global memory is read from here on
    pdl_wait();
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = p.offsets[i];
    if (!WGRAD) {
        __syncthreads();
        if (warp == 0) bucket_odd_prefix(s_off, p.E, s_q, lane);
    } else if (p.rows_used) {
        // (the weight gradients do not use the odd-bucket prefix: its array holds each
        // bucket's k-block count instead; the host passes rows_used only below 2^16 k-blocks)
        for (int i = threadIdx.x; i < p.E; i += blockDim.x) s_q[i] = (uint16_t)((p.rows_used[i] + BK - 1) / BK);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive or complete_tx
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = WGRAD ? p.E * p.m_tiles * p.n_tiles : pairs_before(s_off, s_q, p.E) * p.n_tiles;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs): own A rows, own half of B
        if (lane == 0) {
            uint32_t s = 0, ph = 0;   // ring position: the stage, and the phase of its barriers
            bool ok = true;
            for (int tile = cluster_id; tile < num_tiles && ok; tile += nclusters) {
                const PairTile t = decode_pair_tile<WGRAD>(p, s_off, s_q, tile);
                const int mr = t.m0 + (int)rank * P_HALF;   // this CTA's rows of the tile
                const int nh = t.n0 + (int)rank * P_HALF;   // this CTA's half of B's columns
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(empty + s, ph ^ 1, p.err)) { ok = false; break; }
                    const uint32_t sa = smem_u32(smem + s * P_STAGE_BYTES);
                    const uint32_t sb = sa + P_A_BYTES;
                    const uint32_t fb = map_to_rank(smem_u32(full + s), 0);
                    if (leader) mbar_expect_tx(full + s, 2 * P_STAGE_BYTES);
                    const int k0 = kb * BK;
                    if (!A_MN) {
                        tma_load_2d_pair(sa, &tmA, k0, WGRAD ? t.row0 + (mr - t.m0) : mr, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < P_HALF / 64; ++j)
                            tma_load_2d_pair(sa + j * (BK * 128), &tmA, mr + 64 * j, t.row0 + k0, fb);
                    }
                    if (!B_MN) {
                        tma_load_2d_pair(sb, &tmB, k0, t.e * p.N + nh, fb);
                    } else if (WGRAD) {
#pragma unroll
                        for (int j = 0; j < P_HALF / 64; ++j)
                            tma_load_2d_pair(sb + j * (BK * 128), &tmB, nh + 64 * j, t.row0 + k0, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < P_HALF / 64; ++j)
                            tma_load_2d_pair(sb + j * (BK * 128), &tmB, nh + 64 * j, t.e * p.K + k0, fb);
                    }
                    if (++s == P_STAGES) { s = 0; ph ^= 1; }
                }
            }
            if (!ok) *s_fail = 1;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread of the leader CTA drives the pair
        if (leader && lane == 0) {
            const uint32_t idesc = idesc_bf16(P_BM, BN, A_MN, B_MN);
            // The operands' descriptors at stage 0, k = 0. The start-address field counts 16-byte
            // units, so a stage and a K step of UMMA_K advance it by constants. This keeps the
            // issuing thread's work per k-block small: its instruction latency is on the
            // tensor pipe's critical path.
            const uint32_t s0 = smem_u32(smem);
            const uint64_t a_desc0 = A_MN ? make_desc(s0, BK * 128, 1024) : make_desc(s0, 16, 1024);
            const uint64_t b_desc0 = B_MN ? make_desc(s0 + P_A_BYTES, BK * 128, 1024) : make_desc(s0 + P_A_BYTES, 16, 1024);
            constexpr uint32_t A_KSTEP = (A_MN ? UMMA_K * 128 : UMMA_K * 2) >> 4;
            constexpr uint32_t B_KSTEP = (B_MN ? UMMA_K * 128 : UMMA_K * 2) >> 4;
            constexpr uint32_t STAGE_STEP = P_STAGE_BYTES >> 4;
            uint32_t s = 0, ph = 0, soff = 0, tl = 0;   // ring stage, its phase, its descriptor offset
            bool ok = true;
            for (int tile = cluster_id; tile < num_tiles && ok; tile += nclusters) {
                const PairTile t = decode_pair_tile<WGRAD>(p, s_off, s_q, tile);
                if (t.kblocks == 0) continue;
                const int buf = tl & 1;
                const uint32_t aph = (tl >> 1) & 1;
                ++tl;
                if (!mbar_wait(tempty + buf, aph ^ 1, p.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < t.kblocks; ++kb) {
                    if (!mbar_wait(full + s, ph, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + soff, bd = b_desc0 + soff;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_pair(d_tmem, ad + kk * A_KSTEP, bd + kk * B_KSTEP, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    commit_pair_both(empty + s);   // frees the stage in both CTAs
                    if (++s == P_STAGES) { s = 0; ph ^= 1; soff = 0; } else { soff += STAGE_STEP; }
                }
                if (!ok) break;
                commit_pair_both(tfull + buf);     // both CTAs' accumulator rows are ready
            }
            if (!ok) *s_fail = 1;
            commit_pair_local(drain);
            mbar_wait(drain, 0, p.err);
        }
    } else {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the tile
        const int quarter = warp & 3;
        const int grp = (warp - 2) >> 2;
        const int c_lo = 32 * (grp * (CHUNKS / WPQ) + min(grp, CHUNKS % WPQ));
        const int COLS = 32 * (CHUNKS / WPQ + (grp < CHUNKS % WPQ ? 1 : 0));
        Stager st{smem_u32(stg_smem + (warp - 2) * 2 * STG_BYTES), 0};
        constexpr int NB = pair_ffn1_nb<KIND>();
        Stager2<NB> st2{smem_u32(stg_smem + (warp - 2) * 2 * NB * STG_BYTES), 0};   // Ffn1 only
        const uint32_t tempty_leader[2] = {map_to_rank(smem_u32(tempty), 0), map_to_rank(smem_u32(tempty + 1), 0)};
        uint32_t tl = 0;
        for (int tile = cluster_id; tile < num_tiles; tile += nclusters) {
            const PairTile pt = decode_pair_tile<WGRAD>(p, s_off, s_q, tile);
            Tile t;
            t.e = pt.e; t.n0 = pt.n0; t.row0 = pt.row0; t.kblocks = pt.kblocks;
            t.m0 = pt.m0 + (int)rank * P_HALF;  // this CTA's rows
            const int row_in_tile = quarter * 32 + lane;
            if (t.kblocks == 0) {
                if (KIND == kGemmWgrad) {
                    const int y = t.m0 + quarter * 32;
                    const int cols = min(COLS, p.N - (t.n0 + c_lo));
                    if (y < p.M && cols > 0)
                        st.store_zero(lane, st.acquire(lane), &tmO0, t.n0 + c_lo, (cols + 31) / 32, t.e * p.M + y);
                }
                if (KIND == kGemmWgradF32) {
                    const int m = t.m0 + row_in_tile;
                    for (int c = c_lo; c < c_lo + COLS && m < p.M; c += 32)
                        for (int i = 0; i < 32; i += 4)
                            if (t.n0 + c + i < p.N)
                                *reinterpret_cast<float4*>(p.outf + ((size_t)t.e * p.M + m) * p.N + t.n0 + c + i) =
                                    make_float4(0.f, 0.f, 0.f, 0.f);
                }
                continue;
            }
            const int buf = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            ++tl;
            // the second half of an odd bucket's last tile lies past the bucket: computed by the
            // pair's MMAs, not stored (its accumulator is only released)
            const bool dead = !WGRAD && t.m0 >= pt.end;
            const size_t aux_row0 = (size_t)(t.m0 + quarter * 32 + (lane >> 2));
            // side input (bias row, or dH's saved GELU'(A)) of the first chunk, fetched while the
            // accumulator is produced; each later chunk's is fetched one chunk ahead
            Raw32 next;
            if (!dead && t.n0 + c_lo < p.N) {
                if (has_bias<KIND>()) load_raw32(next, p.bias + (size_t)t.e * p.N + t.n0 + c_lo);
                if (AUX) load_aux32<KIND>(next, p, aux_row0, t.n0 + c_lo, lane);
            }
            if (!mbar_wait(tfull + buf, aph, p.err)) break;
            tc_fence_after();
            if (dead) {
                tc_fence_before();
                if (leader) mbar_arrive(tempty + buf);
                else mbar_arrive_cluster(tempty_leader[buf]);
                if (*s_fail) break;
                continue;
            }
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN;
            // with PREFETCH the TMEM load of chunk c + 32 is in flight while chunk c is processed
            uint32_t acc[32];
            if (PREFETCH && t.n0 + c_lo < p.N) tmem_ld32(taddr + c_lo, acc);
            for (int c = c_lo; c < c_lo + COLS; c += 32) {
                if (t.n0 + c >= p.N) break;
                const int n = t.n0 + c;
                const Raw32 cur = next;
                const bool more = c + 32 < c_lo + COLS && n + 32 < p.N;
                if (more && has_bias<KIND>()) load_raw32(next, p.bias + (size_t)t.e * p.N + n + 32);
                if (more && AUX) load_aux32<KIND>(next, p, aux_row0, n + 32, lane);
                if (!PREFETCH) tmem_ld32(taddr + c, acc);
                tmem_ld_wait_regs(acc);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
                if (PREFETCH && more) tmem_ld32(taddr + c + 32, acc);
                const int y = t.m0 + quarter * 32;
                if (KIND == kGemmWgradF32) {
                    // each lane writes its row's 32 fp32 values (128 contiguous bytes)
                    const int m = y + lane;
                    if (m < p.M) {
                        float* dst = p.outf + ((size_t)t.e * p.M + m) * p.N + n;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            if (n + i < p.N)
                                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                } else if (KIND == kGemmWgrad) {
                    const uint32_t b = st.acquire(lane);
                    if (y < p.M) st.store(lane, b, v, &tmO0, n, t.e * p.M + y);
                } else if (KIND == kGemmFfn1 || KIND == kGemmFfn2) {
                    float bv[32];
                    unpack_raw32(cur, bv);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) upk2(add2(pk2(v[i], v[i + 1]), pk2(bv[i], bv[i + 1])), v[i], v[i + 1]);
                    if (KIND == kGemmFfn1) {
                        // H = GELU(A) for the second GEMM, GELU'(A) saved for the backward
                        const uint32_t b = st2.acquire(lane);
                        st2.store_gelu(lane, b, v, &tmO0, &tmO1, n, y);
                    } else {
                        const uint32_t b = st.acquire(lane);
                        st.store(lane, b, v, &tmO0, n, y);
                    }
                } else if (AUX) {
                    // the side input arrived coalesced (lane l: rows (l>>2)+8i, 16-byte segment
                    // l&3); the staging buffer turns it into this lane's row
                    const uint32_t b = st.acquire(lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i) sts128(sw64_addr(b, (lane >> 2) + 8 * i, lane & 3), cur.q[i]);
                    __syncwarp();
                    float a[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) unpack8(lds128(sw64_addr(b, lane, j)), a + 8 * j);
                    __syncwarp();
                    if (KIND == kGemmDH) {
#pragma unroll
                        for (int i = 0; i < 32; i += 2)   // a = GELU'(A) saved by the forward
                            upk2(mul2(pk2(v[i], v[i + 1]), pk2(a[i], a[i + 1])), v[i], v[i + 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] += a[i];  // accumulate into aux (= out0)
                    }
                    st.store(lane, b, v, &tmO0, n, y);
                    if (KIND == kGemmDH && p.colsum) {
                        // db1 partial of this lane quarter (32 rows) from the staged dA chunk
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
            if (leader) mbar_arrive(tempty + buf);
            else mbar_arrive_cluster(tempty_leader[buf]);
            if (*s_fail) break;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // all work of both CTAs is done before the pair releases its TMEM
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

template <int KIND>
constexpr size_t pair_smem_bytes() {
    return 1024 + (size_t)pair_stages<KIND>() * P_STAGE_BYTES + pair_epi_bytes<KIND>() + 16 * sizeof(uint64_t) +
           16 + kMaxOffsets * (sizeof(int) + sizeof(uint16_t));
}
static_assert(pair_smem_bytes<kGemmFfn1>() <= 227 * 1024 && pair_smem_bytes<kGemmFfn2>() <= 227 * 1024,
              "shared memory per CTA");

template <int KIND, bool A_MN, bool B_MN>
cudaError_t launch_pair(const TcParams& p, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o0,
                        const CUtensorMap& o1, int clusters, cudaStream_t s) {
    constexpr size_t kPairSmemBytes = pair_smem_bytes<KIND>();
    auto kern = tc_gemm_pair_kernel<KIND, A_MN, B_MN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmemBytes);
    if (e != cudaSuccess) return e;
    launch_pdl(kern, 2 * clusters, pair_threads<KIND>(), kPairSmemBytes, s, p, a, b, o0, o1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_gemm_tc_pair(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s) {
    if (a.rows_capacity == 0) return cudaSuccess;
    if (a.rows_capacity % BM != 0) return cudaErrorInvalidValue;  // buckets are 128-row aligned
    TcParams p{};
    p.kind = a.kind;
    p.offsets = a.offsets;
    const int rows_valid = a.rows_valid > 0 ? a.rows_valid : a.rows_capacity;
    p.E = a.E; p.N = a.N; p.K = a.K; p.M = rows_valid;
    p.n_tiles = ceil_div(a.N, BN);
    p.m_tiles = ceil_div(a.rows_capacity, P_BM);   // (grid sizing) pair tiles per column block, at most
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.aux = static_cast<const __nv_bfloat16*>(a.aux);
    p.out0 = static_cast<__nv_bfloat16*>(a.out0);
    p.out1 = static_cast<__nv_bfloat16*>(a.out1);
    p.colsum = a.colsum;
    p.err = device_error_word();
    CUtensorMap ta, tb, to0, to1;
    // A: activations [rows, K], each CTA its own 128 rows
    if (!make_map(&ta, a.A, (uint64_t)a.K, (uint64_t)a.rows_capacity, P_HALF)) return cudaErrorInvalidValue;
    if (a.sBn != 1) {
        // B(n, k) = W[e*N + n][k], K-major: each CTA its own 128 of the tile's 256 columns
        if (!make_map(&tb, a.B, (uint64_t)a.K, (uint64_t)a.E * a.N, P_HALF)) return cudaErrorInvalidValue;
    } else {
        // B(n, k) = W[e*K + k][n], N-major: boxes of 64 n x 64 k
        if (!make_map(&tb, a.B, (uint64_t)a.N, (uint64_t)a.E * a.K, BK)) return cudaErrorInvalidValue;
    }
    // stores to rows that do not exist (rows_valid < rows_capacity) fall outside the map
    if (!make_map_ex(&to0, a.out0, (uint64_t)a.N, (uint64_t)rows_valid, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (a.kind == kGemmFfn1) {
        if (!make_map_ex(&to1, a.out1, (uint64_t)a.N, (uint64_t)a.rows_capacity, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        to1 = to0;
    }
    const long long tiles = (long long)p.m_tiles * p.n_tiles;
    const int clusters = (int)std::max(1LL, std::min<long long>(tiles, num_sms() / 2));
    switch (a.kind) {
        case kGemmFfn1: return launch_pair<kGemmFfn1, false, false>(p, ta, tb, to0, to1, clusters, s);
        case kGemmFfn2: return launch_pair<kGemmFfn2, false, false>(p, ta, tb, to0, to1, clusters, s);
        case kGemmDH: return launch_pair<kGemmDH, false, true>(p, ta, tb, to0, to1, clusters, s);
        case kGemmDX: return launch_pair<kGemmDX, false, true>(p, ta, tb, to0, to1, clusters, s);
        case kGemmAccum: return launch_pair<kGemmAccum, false, true>(p, ta, tb, to0, to1, clusters, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wgrad_tc_pair(const moe_config_t& c, const WgradArgs& a, cudaStream_t s) {
    TcParams p{};
    p.kind = a.f32 ? kGemmWgradF32 : kGemmWgrad;
    p.offsets = a.offsets;
    p.E = a.E; p.N = a.N; p.M = a.M; p.K = 0;
    p.n_tiles = ceil_div(a.N, BN);
    p.m_tiles = ceil_div(a.M, P_BM);
    p.out0 = a.f32 ? nullptr : static_cast<__nv_bfloat16*>(a.C);
    p.outf = a.f32 ? static_cast<float*>(a.C) : nullptr;
    p.rows_used = (!a.f32 && a.rows_used && (long long)c.rows_capacity / BK < 65536) ? a.rows_used : nullptr;
    p.err = device_error_word();
    CUtensorMap ta, tb, to0;
    const uint64_t rows_p = (uint64_t)std::max(a.rows_p > 0 ? a.rows_p : c.rows_capacity, 1);
    const uint64_t rows_q = (uint64_t)std::max(a.rows_q > 0 ? a.rows_q : c.rows_capacity, 1);
    if (!make_map(&ta, a.P, (uint64_t)a.M, rows_p, BK)) return cudaErrorInvalidValue;
    if (!make_map(&tb, a.Q, (uint64_t)a.N, rows_q, BK)) return cudaErrorInvalidValue;
    if (a.f32) {
        to0 = ta;   // unused: the fp32 epilogue writes from registers
    } else if (!make_map_ex(&to0, a.C, (uint64_t)a.N, (uint64_t)a.E * a.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) {
        return cudaErrorInvalidValue;
    }
    const long long tiles = (long long)a.E * p.m_tiles * p.n_tiles;
    const int clusters = (int)std::max(1LL, std::min<long long>(tiles, num_sms() / 2));
    if (a.f32) return launch_pair<kGemmWgradF32, true, true>(p, ta, tb, to0, to0, clusters, s);
    return launch_pair<kGemmWgrad, true, true>(p, ta, tb, to0, to0, clusters, s);
}

}  // namespace moe
