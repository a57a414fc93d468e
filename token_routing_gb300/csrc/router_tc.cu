// Router on the tensor cores: the gate linear z = x Wg^T as a tcgen05 GEMM (bf16 operands
// staged by TMA, fp32 accumulation in TMEM), fused with the bias, the top-k selection
// (ties -> lower expert id), the softmax over the k selected logits divided by the
// temperature, and the per-expert counts.
//
// "Native MoE training system PithTrain", section 4.1 (gate, torch.topk, softmax over the
// selected values); "Expert Parallelism: Scaling Mixture-of-Experts Models", section 2.2
// (softmax(gate(x) / temperature), top-8 pre-selection) and section 5.5 (routing in FP32:
// the logits stay fp32 from the accumulator to the softmax).
//
// One CTA per 128-token tile: warp 0 streams x and Wg tiles with TMA, warp 1 issues the
// MMAs (N = E rounded up to 32), and G groups of four epilogue warps (one per TMEM lane
// quarter) read the logits from TMEM. With k = E one group takes the softmax over all E per
// token. For top-k, group g takes its share of the 32-expert chunks (chunks g, g + G, ...;
// G = min(4, chunks)), and the groups' results meet through shared memory:
//   * k = 8: value-only sorting networks give each token's 8 largest logits; the experts at or
//     above the 8th go to their slots by rank, and a token with tied logits there takes the
//     exact (logit, id) order over all its experts;
//   * other k: each group keeps a sorted top-k list per token, and group 0 merges the G lists.
// In each CTA the selection starts once the whole x tile has been read.
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int RBM = 128;
constexpr int RBK = 64;
constexpr int RMAX_STAGES = 12;              // ring depth: as many stages as fit in ~200 KB
constexpr int RSMEM_BUDGET = 200 * 1024;
// warps 0 (TMA) and 1 (MMA) plus G groups of four epilogue warps
__host__ __device__ constexpr int route_threads(int G) { return 64 + 128 * G; }

struct RouteTcParams {
    int T, d, E, E_pad, stages;
    int rows;          // tokens per tile (at most RBM)
    int tiles;         // ceil(T / rows); the CTAs take tiles blockIdx.x, + gridDim.x, ...
    float inv_temp;
    float noise_std;
    uint32_t noise_seed;
    const float* bg;
    int32_t* idx;
    float* w;
    int32_t* counts;
    float* logits;   // [T, E] or null
    const float* noise;   // [E, T] N(0,1) draws, or null (no noise)
    int* err;
};

__host__ __device__ constexpr int route_stage_bytes(int E_pad) { return RBM * RBK * 2 + E_pad * RBK * 2; }

// The routing-noise draws of experts c .. c + 31 for one token ([E, T] layout; zero past E or
// without a token), all loaded before the chunk's stores so that the 32 loads overlap instead
// of each waiting behind the previous expert's stores.
__device__ __forceinline__ void load_noise32(const float* __restrict__ noise, int T, int E, int c, int tok,
                                             bool live, float (&nz)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) nz[i] = (live && c + i < E) ? __ldg(noise + (size_t)(c + i) * T + tok) : 0.f;
}

// N consecutive logits of a token (columns c .. c + N - 1 of its TMEM row: bias, optional
// noise and logits output) inserted into its list sorted by (logit desc, id asc). A new expert
// (ids arrive in ascending order) never displaces an equal logit; once it has displaced an
// entry, the rest of the list shifts down one slot (each pushed entry comes before the next in
// that order, equal logits included).
template <int K, int N, bool NOISE>
__device__ __forceinline__ void select_cols(const RouteTcParams& p, const uint32_t (&r)[N], const float (&nz)[N],
                                            int c, int tok, const float* s_bias, float (&tv)[K], int (&te)[K]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        int e = c + i;
        if (e < p.E) {
            float v = __uint_as_float(r[i]) + s_bias[e];
            if (NOISE && tok < p.T) v = fmaf(p.noise_std, nz[i], v);
            if (p.logits && tok < p.T) p.logits[(size_t)tok * p.E + e] = v;
            bool moved = false;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (moved || te[j] < 0 || v > tv[j]) {
                    const float ov = tv[j];
                    const int oe = te[j];
                    tv[j] = v; te[j] = e;
                    v = ov; e = oe;
                    moved = true;
                }
            }
        }
    }
}

// One 32-expert chunk of a token's logits into its top-k list. Without noise, one 32-column
// TMEM load; with noise, two halves of 16 columns and 16 draws each, so that the draws do
// not add to the live registers of the 32-column path (a 576-thread block allows 96 per
// thread; more spilled the lists to local memory in the selection).
template <int K>
__device__ __forceinline__ void select_chunk(const RouteTcParams& p, uint32_t taddr, int c, int tok,
                                             const float* s_bias, float (&tv)[K], int (&te)[K]) {
    if (p.noise) {
#pragma unroll 1
        for (int h = 0; h < 32; h += 16) {
            float nz[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                nz[i] = (tok < p.T && c + h + i < p.E) ? __ldg(p.noise + (size_t)(c + h + i) * p.T + tok) : 0.f;
            uint32_t r[16];
            tmem_ld16(taddr + c + h, r);
            tmem_ld_wait();
            select_cols<K, 16, true>(p, r, nz, c + h, tok, s_bias, tv, te);
        }
    } else {
        uint32_t r[32];
        const float nz[32] = {};
        tmem_ld32(taddr + c, r);
        tmem_ld_wait();
        select_cols<K, 32, false>(p, r, nz, c, tok, s_bias, tv, te);
    }
}

// ---- top-8 in two passes (k = 8)
//
// Pass 1 finds the token's 8th-largest logit theta with value-only sorting networks (a
// comparator is one max and one min). Every expert of the top 8 then has a logit >= theta, and
// any expert below theta has 8 larger ones, so pass 2 collects the experts with logit >= theta
// (8 of them unless logits tie at theta) and sorts only those by (logit desc, id asc).
//
// A (logit, expert) pair as one 64-bit key whose unsigned order is the selection order: the
// logit's bits mapped to an order-preserving integer in the high word, the complement of the
// expert id in the low word (equal logits: the lower id has the larger key). Key 0 lies below
// every real logit and marks an empty slot (expert -1). -0 is folded into +0 first so that
// the two compare equal, as the logits do.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
    uint32_t u = __float_as_uint(v + 0.0f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)u << 32) | (uint32_t)~e;
}
__device__ __forceinline__ float key_logit(uint64_t k) {
    const uint32_t u = (uint32_t)(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
__device__ __forceinline__ int key_expert(uint64_t k) { return (int)~(uint32_t)k; }

// comparators: a >= b afterwards
__device__ __forceinline__ uint64_t vmax(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ float vmax(float a, float b) { return fmaxf(a, b); }
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
    const uint64_t hi = a > b ? a : b;
    b = a > b ? b : a;
    a = hi;
}
__device__ __forceinline__ void cas_desc(float& a, float& b) {
    const float hi = fmaxf(a, b);
    b = fminf(a, b);
    a = hi;
}

// Batcher's odd-even merge sort of 8 values, descending (19 comparators in 6 layers).
template <typename V>
__device__ __forceinline__ void sort8_desc(V (&k)[8]) {
    cas_desc(k[0], k[1]); cas_desc(k[2], k[3]); cas_desc(k[4], k[5]); cas_desc(k[6], k[7]);
    cas_desc(k[0], k[2]); cas_desc(k[1], k[3]); cas_desc(k[4], k[6]); cas_desc(k[5], k[7]);
    cas_desc(k[1], k[2]); cas_desc(k[5], k[6]);
    cas_desc(k[0], k[4]); cas_desc(k[1], k[5]); cas_desc(k[2], k[6]); cas_desc(k[3], k[7]);
    cas_desc(k[2], k[4]); cas_desc(k[3], k[5]);
    cas_desc(k[1], k[2]); cas_desc(k[3], k[4]); cas_desc(k[5], k[6]);
}

// The 8 largest of two descending lists, descending, into r: the pairwise maxima of r and the
// reversed s form a bitonic sequence that holds them, and three half-cleaner layers sort it.
template <typename V>
__device__ __forceinline__ void merge8_desc(V (&r)[8], const V (&s)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = vmax(r[i], s[7 - i]);
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if ((i & d) == 0) cas_desc(r[i], r[i + d]);
}

// The routing logit of expert e for a token from its accumulator column: bias, then noise.
// Both passes compute it with this one expression, so they see the same bits.
template <bool NOISE>
__device__ __forceinline__ float route_logit(const RouteTcParams& p, uint32_t acc, float nz, int e, int tok,
                                             const float* s_bias) {
    float v = __uint_as_float(acc) + s_bias[e];
    if (NOISE && tok < p.T) v = fmaf(p.noise_std, nz, v);
    return v;
}

// Accumulator columns c .. c + 15 of the thread's token, and their noise draws.
__device__ __forceinline__ void load_cols16(const RouteTcParams& p, uint32_t taddr, int c, int tok,
                                            uint32_t (&r)[16], float (&nz)[16]) {
    if (p.noise) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            nz[i] = (tok < p.T && c + i < p.E) ? __ldg(p.noise + (size_t)(c + i) * p.T + tok) : 0.f;
    }
    tmem_ld16(taddr + c, r);
    tmem_ld_wait();
}

// Pass 1 over experts c .. c + 15: their logits into the token's 8 largest values so far
// (experts past E count as -inf), into its row of the staged logits s_v ([E][RBM]) and into
// the logits output.
template <bool NOISE>
__device__ __forceinline__ void top8_values16(const RouteTcParams& p, const uint32_t (&r)[16], const float (&nz)[16],
                                              int c, int tok, int row, const float* s_bias, float* s_v,
                                              float (&top)[8]) {
#pragma unroll
    for (int g = 0; g < 16; g += 8) {
        float k[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = c + g + i;
            k[i] = -INFINITY;
            if (e < p.E) {
                k[i] = route_logit<NOISE>(p, r[g + i], nz[g + i], e, tok, s_bias);
                s_v[e * RBM + row] = k[i];
                if (p.logits && tok < p.T) p.logits[(size_t)tok * p.E + e] = k[i];
            }
        }
        sort8_desc(k);
        merge8_desc(top, k);
    }
}

// Softmax over a token's k selected logits (tv[0] the largest), its indices and weights, and
// its counts in the CTA's histogram.
template <int K>
__device__ __forceinline__ void route_finish(const RouteTcParams& p, int tok, const float (&tv)[K],
                                             const int (&te)[K], int* s_cnt) {
    float pr[K], s = 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j) { pr[j] = expf((tv[j] - tv[0]) * p.inv_temp); s += pr[j]; }
    const float inv = 1.f / s;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        p.idx[(size_t)tok * K + j] = te[j];
        p.w[(size_t)tok * K + j] = pr[j] * inv;
        if (te[j] >= 0) atomicAdd(&s_cnt[te[j]], 1);
    }
}

__device__ __forceinline__ void epilogue_bar_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int K, int G>
__global__ void __launch_bounds__(route_threads(G), 1)
route_tc_kernel(const RouteTcParams p, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmW) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = route_stage_bytes(p.E_pad);
    const int RSTAGES = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RSTAGES * stage_bytes);
    uint64_t* empty = full + RMAX_STAGES;
    uint64_t* tfull = empty + RMAX_STAGES;   // [2]: accumulator buffers
    uint64_t* tempty = tfull + 2;            // [2]
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* s_cnt = reinterpret_cast<int*>(tmem_slot + 4);
    float* s_bias = reinterpret_cast<float*>(s_cnt + MOE_MAX_EXPERTS);
    uint8_t* s_scratch = reinterpret_cast<uint8_t*>(s_bias + MOE_MAX_EXPERTS);   // top-k merge lists
    __shared__ int s_fail;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = (p.d + RBK - 1) / RBK;
    const uint32_t ncols = p.E_pad <= 32 ? 32 : p.E_pad <= 64 ? 64 : p.E_pad <= 128 ? 128 : 256;
    // Top-k with k < 8 may take several tiles per CTA: two accumulators, so that the MMAs of a
    // tile run while the epilogue selects over the previous one. The k = 8 and k = E paths
    // take one tile per CTA and stage their work over the operand ring.
    constexpr bool MULTI = K > 0 && K < 8;
    const uint32_t nalloc = MULTI ? 2 * ncols : ncols;

    for (int e = threadIdx.x; e < MOE_MAX_EXPERTS; e += blockDim.x) s_cnt[e] = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(tfull + b, 1); mbar_init(tempty + b, 128 * G); }
        mbar_init(drain, 1);
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, nalloc);
    // everything above touches only this CTA's shared memory and TMEM, and overlaps the
    // previous kernel's tail; global memory is read from here on
    pdl_wait();
    for (int e = threadIdx.x; e < MOE_MAX_EXPERTS; e += blockDim.x) s_bias[e] = (p.bg && e < p.E) ? p.bg[e] : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // Each tile starts its walk along d at its own k-block (tile index mod the k-block
            // count) and wraps around: otherwise every CTA reads the same 128-byte column block
            // of its rows, and of Wg, at the same time. `it` counts the loads issued.
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
                const int kb0 = tile % kblocks;
                for (int kb = 0; kb < kblocks; ++kb) {
                    const int s = it % RSTAGES;
                    const uint32_t ph = (it / RSTAGES) & 1;
                    if (!mbar_wait(empty + s, ph ^ 1, p.err)) { ok = false; break; }
                    const uint32_t sa = smem_u32(smem + s * stage_bytes);
                    const int kc = kb + kb0 < kblocks ? kb + kb0 : kb + kb0 - kblocks;
                    mbar_expect_tx(full + s, p.rows * RBK * 2 + p.E_pad * RBK * 2);
                    tma_load_2d(sa, &tmX, kc * RBK, tile * p.rows, full + s);
                    tma_load_2d(sa + RBM * RBK * 2, &tmW, kc * RBK, 0, full + s);
                    ++it;
                }
            }
            if (!ok) {
                s_fail = 1;
                for (int j = it > RSTAGES ? it - RSTAGES : 0; j < it; ++j)
                    mbar_wait(full + j % RSTAGES, (j / RSTAGES) & 1, p.err);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(RBM, p.E_pad, false, false);
            bool ok = true;
            int it = 0, tl = 0;   // loads consumed, tiles started
            for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++tl) {
                const int buf = tl & 1;
                if (!mbar_wait(tempty + buf, ((tl >> 1) & 1) ^ 1, p.err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * ncols;
                for (int kb = 0; kb < kblocks; ++kb) {
                    const int s = it % RSTAGES;
                    const uint32_t ph = (it / RSTAGES) & 1;
                    if (!mbar_wait(full + s, ph, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * stage_bytes);
                    const uint32_t sb = sa + RBM * RBK * 2;
#pragma unroll
                    for (int kk = 0; kk < RBK / 16; ++kk)
                        tc_mma(d_tmem, make_desc(sa + kk * 32, 16, 1024), make_desc(sb + kk * 32, 16, 1024), idesc,
                               (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(empty + s);
                    ++it;
                }
                if (ok) tc_commit(tfull + buf);
            }
            if (!ok) s_fail = 1;
            tc_commit(drain);
            mbar_wait(drain, 0, p.err);
        }
    } else {
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        // every epilogue thread runs every tile, with no early exit: the top-k merge meets at a
        // named barrier (a wait that ran out leaves the tile's lists empty)
        int tl = 0;
        for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tl) {
            const int buf = tl & 1;
            const uint32_t aph = (tl >> 1) & 1;
            const int tok = row < p.rows ? tile * p.rows + row : p.T;   // rows beyond the tile: no token
            if constexpr (K == 0) {
                // dense soft routing: w[t, e] = softmax(z_t / temp)_e over all E, slot e = expert e.
                // Three passes over the row (max, sum, write). Without noise every pass reads the
                // logits from TMEM; with noise the first pass leaves the noisy logits in the
                // token's own w row (each normal is drawn once) and the later passes read them back.
                if (mbar_wait(tfull + buf, aph, p.err)) {
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * ncols;
                    const bool live = tok < p.T;
                    if (p.noise) {
                        float* wr = p.w + (size_t)(live ? tok : 0) * p.E;
                        float m = -INFINITY;
                        for (int c = 0; c < p.E_pad; c += 32) {   // warp-uniform TMEM loads
                            float nz[32];
                            load_noise32(p.noise, p.T, p.E, c, tok, live, nz);
                            uint32_t r[32];
                            tmem_ld32(taddr + c, r);
                            tmem_ld_wait();
    #pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int e = c + i;
                                if (e < p.E && live) {
                                    const float v = fmaf(p.noise_std, nz[i], __uint_as_float(r[i]) + s_bias[e]);
                                    if (p.logits) p.logits[(size_t)tok * p.E + e] = v;
                                    wr[e] = v;
                                    m = fmaxf(m, v);
                                }
                            }
                        }
                        if (live) {
                            float ssum = 0.f;
                            for (int e = 0; e < p.E; ++e) ssum += expf((wr[e] - m) * p.inv_temp);
                            const float inv = 1.f / ssum;
                            for (int e = 0; e < p.E; ++e) {
                                p.idx[(size_t)tok * p.E + e] = e;
                                wr[e] = expf((wr[e] - m) * p.inv_temp) * inv;
                            }
                        }
                    } else {
                        float m = -INFINITY, ssum = 0.f;
                        for (int pass = 0; pass < 3; ++pass) {
                            const float inv = pass == 2 ? 1.f / ssum : 0.f;
                            for (int c = 0; c < p.E_pad; c += 32) {
                                uint32_t r[32];
                                tmem_ld32(taddr + c, r);
                                tmem_ld_wait();
    #pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const int e = c + i;
                                    if (e < p.E) {
                                        const float v = __uint_as_float(r[i]) + s_bias[e];
                                        if (pass == 0) {
                                            if (p.logits && live) p.logits[(size_t)tok * p.E + e] = v;
                                            m = fmaxf(m, v);
                                        } else if (pass == 1) {
                                            ssum += expf((v - m) * p.inv_temp);
                                        } else if (live) {
                                            p.idx[(size_t)tok * p.E + e] = e;
                                            p.w[(size_t)tok * p.E + e] = expf((v - m) * p.inv_temp) * inv;
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
            } else if constexpr (K == 8) {
                // Shared memory over the operand ring, which the accumulator-full barrier has
                // retired (the host checks that it holds these): the staged logits, the G groups'
                // value lists, each token's 8 largest values, the experts in their slots and the
                // count of logits at or above theta.
                float* s_v = reinterpret_cast<float*>(smem);                   // [E][RBM]
                float* s_f = s_v + (size_t)p.E * RBM;                          // [G][8][RBM]
                float* s_top = s_f + (size_t)G * 8 * RBM;                      // [8][RBM]
                int* s_e = reinterpret_cast<int*>(s_top + 8 * RBM);            // [8][RBM]
                int* s_n = s_e + 8 * RBM;                                      // [RBM]
                const int grp = (warp - 2) >> 2;
                const bool live = tok < p.T;
                const bool ok = mbar_wait(tfull + buf, aph, p.err);
                if (ok) tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * ncols;
                // pass 1: the 8 largest logits of the group's chunks (chunks grp, grp + G, ...)
                float top[8];
    #pragma unroll
                for (int j = 0; j < 8; ++j) top[j] = -INFINITY;
                for (int c = 32 * grp; ok && c < p.E_pad; c += 32 * G) {
    #pragma unroll 1
                    for (int h = c; h < c + 32 && h < p.E; h += 16) {   // warp-uniform bounds
                        uint32_t r[16];
                        float nz[16];
                        load_cols16(p, taddr, h, tok, r, nz);
                        if (p.noise) top8_values16<true>(p, r, nz, h, tok, row, s_bias, s_v, top);
                        else top8_values16<false>(p, r, nz, h, tok, row, s_bias, s_v, top);
                    }
                }
                // the G lists meet in a tree: odd groups hand theirs to the even group below, then
                // group 2 to group 0, which then holds the token's 8 largest logits
                if constexpr (G > 1) {
                    if (grp & 1) {
    #pragma unroll
                        for (int j = 0; j < 8; ++j) s_f[((size_t)grp * 8 + j) * RBM + row] = top[j];
                    }
                    epilogue_bar_sync(128 * G);
                    if (!(grp & 1) && grp + 1 < G) {
                        float o[8];
    #pragma unroll
                        for (int j = 0; j < 8; ++j) o[j] = s_f[((size_t)(grp + 1) * 8 + j) * RBM + row];
                        merge8_desc(top, o);
                    }
                    if constexpr (G > 2) {
                        if (grp == 2) {
    #pragma unroll
                            for (int j = 0; j < 8; ++j) s_f[((size_t)2 * 8 + j) * RBM + row] = top[j];
                        }
                        epilogue_bar_sync(128 * G);
                        if (grp == 0) {
                            float o[8];
    #pragma unroll
                            for (int j = 0; j < 8; ++j) o[j] = s_f[((size_t)2 * 8 + j) * RBM + row];
                            merge8_desc(top, o);
                        }
                    }
                }
                if (grp == 0) {
    #pragma unroll
                    for (int j = 0; j < 8; ++j) s_top[j * RBM + row] = top[j];
                    s_n[row] = 0;
                }
                epilogue_bar_sync(128 * G);
                // pass 2: each expert of the group with logit >= theta = the 8th value goes to slot
                // (number of the 8 values above its logit). With distinct values and exactly 8 such
                // experts that is the order (logit desc); anything else is a tie, found below.
                if (live) {
                    float vt[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j) vt[j] = s_top[j * RBM + row];
                    for (int c = 32 * grp; ok && c < p.E_pad; c += 32 * G) {
                        uint32_t mask = 0;
    #pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c + i < p.E && s_v[(c + i) * RBM + row] >= vt[7]) mask |= 1u << i;
                        while (mask) {
                            const int e = c + __ffs(mask) - 1;
                            mask &= mask - 1;
                            const float v = s_v[e * RBM + row];
                            int slot = 0;
    #pragma unroll
                            for (int j = 0; j < 8; ++j) slot += vt[j] > v ? 1 : 0;
                            if (slot < 8) s_e[slot * RBM + row] = e;
                            atomicAdd(s_n + row, 1);
                        }
                    }
                }
                epilogue_bar_sync(128 * G);
                if (grp == 0 && live) {
                    float tv[8];
                    int te[8];
                    bool tie = s_n[row] != 8;
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        tv[j] = top[j];
                        te[j] = s_e[j * RBM + row];
                        if (j > 0 && top[j] == top[j - 1]) tie = true;
                    }
                    if (tie) {
                        // equal logits in or at the edge of the top 8: the exact order over every
                        // expert's (logit, id) key, from the staged logits
                        uint64_t key[8];
    #pragma unroll
                        for (int j = 0; j < 8; ++j) key[j] = 0;
                        for (int c = 0; c < p.E; c += 8) {
                            uint64_t k[8];
    #pragma unroll
                            for (int i = 0; i < 8; ++i)
                                k[i] = c + i < p.E ? sel_key(s_v[(c + i) * RBM + row], c + i) : 0;
                            sort8_desc(k);
                            merge8_desc(key, k);
                        }
    #pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            tv[j] = key[j] ? key_logit(key[j]) : -INFINITY;
                            te[j] = key_expert(key[j]);
                        }
                    }
                    route_finish<8>(p, tok, tv, te, s_cnt);
                }
            } else {
                const int grp = (warp - 2) >> 2;
                float tv[K];
                int te[K];
    #pragma unroll
                for (int j = 0; j < K; ++j) { tv[j] = -INFINITY; te[j] = -1; }
                const bool ok = mbar_wait(tfull + buf, aph, p.err);
                if (ok) tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * ncols;
                for (int c = 32 * grp; ok && c < p.E_pad; c += 32 * G) {
                    select_chunk<K>(p, taddr, c, tok, s_bias, tv, te);
                }
                // the accumulator is read: the MMAs of the tile after next may overwrite it
                tc_fence_before();
                mbar_arrive(tempty + buf);
                if constexpr (G == 1) {
                    if (tok < p.T) route_finish<K>(p, tok, tv, te, s_cnt);
                } else {
                    // The G partial lists of each token go to shared memory, in one of two buffers
                    // by tile parity: group 0 reads a tile's buffer before it reaches the next
                    // tile's barrier, which the other groups must pass before they write that
                    // buffer again (a wait that ran out leaves empty lists, and the id check below
                    // keeps them out of the counts).
                    float* s_v = reinterpret_cast<float*>(s_scratch) + (size_t)(tl & 1) * 2 * G * RBM * K;   // [G][RBM][K]
                    int* s_i = reinterpret_cast<int*>(s_v + (size_t)G * RBM * K);                            // [G][RBM][K]
    #pragma unroll
                    for (int j = 0; j < K; ++j) {
                        s_v[((size_t)grp * RBM + row) * K + j] = tv[j];
                        s_i[((size_t)grp * RBM + row) * K + j] = te[j];
                    }
                    epilogue_bar_sync(128 * G);
                    if (grp == 0) {
                        // Merge of G lists sorted by (logit desc, id asc): take the larger head, the
                        // lower expert id on equal logits, so the result is the top-k of all E.
                        int head[G];
    #pragma unroll
                        for (int g = 0; g < G; ++g) head[g] = 0;
    #pragma unroll
                        for (int j = 0; j < K; ++j) {
                            float bv = -INFINITY;
                            int bi = -1, bg = 0;
    #pragma unroll
                            for (int g = 0; g < G; ++g) {
                                if (head[g] < K) {
                                    const float v = s_v[((size_t)g * RBM + row) * K + head[g]];
                                    const int i = s_i[((size_t)g * RBM + row) * K + head[g]];
                                    if (i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi))) { bv = v; bi = i; bg = g; }
                                }
                            }
                            tv[j] = bv;
                            te[j] = bi;
    #pragma unroll
                            for (int g = 0; g < G; ++g) head[g] += (g == bg && bi >= 0) ? 1 : 0;
                        }
                        if (tok < p.T) route_finish<K>(p, tok, tv, te, s_cnt);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
        if (s_cnt[e]) atomicAdd(p.counts + e, s_cnt[e]);
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, nalloc);
    }
}

template <int K, int G>
cudaError_t launch_kg(const RouteTcParams& p, const CUtensorMap& tx, const CUtensorMap& tw, size_t smem, int grid,
                      cudaStream_t s) {
    auto kern = route_tc_kernel<K, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    launch_pdl(kern, dim3(grid), dim3(route_threads(G)), smem, s, p, tx, tw);
    count_launch();
    return cudaGetLastError();
}

// Epilogue groups: one per 32-expert chunk up to four (dense routing: one).
__host__ __device__ constexpr int route_groups(int K, int E_pad) {
    return K == 0 ? 1 : (E_pad / 32 < 4 ? (E_pad / 32 < 1 ? 1 : E_pad / 32) : 4);
}

template <int K>
cudaError_t launch_k(const RouteTcParams& p, const CUtensorMap& tx, const CUtensorMap& tw, size_t smem, int grid,
                     cudaStream_t s) {
    if constexpr (K == 0) {
        return launch_kg<0, 1>(p, tx, tw, smem, grid, s);
    } else {
        switch (route_groups(K, p.E_pad)) {
            case 1: return launch_kg<K, 1>(p, tx, tw, smem, grid, s);
            case 2: return launch_kg<K, 2>(p, tx, tw, smem, grid, s);
            case 3: return launch_kg<K, 3>(p, tx, tw, smem, grid, s);
            default: return launch_kg<K, 4>(p, tx, tw, smem, grid, s);
        }
    }
}

}  // namespace

bool tc_route_supported(const moe_config_t& c) { return c.dtype == MOE_BF16 && c.d % 64 == 0; }

cudaError_t launch_route_tc(const moe_config_t& c, const void* x, const void* Wg, const float* bg,
                            int32_t* idx, float* w, int32_t* counts, float* logits, const float* noise,
                            cudaStream_t s) {
    RouteTcParams p{};
    p.T = c.T; p.d = c.d; p.E = c.E;
    p.E_pad = (c.E + 31) / 32 * 32;
    p.inv_temp = 1.0f / c.temperature;
    p.noise_std = c.noise_std;
    p.noise_seed = c.noise_seed;
    p.bg = c.has_gate_bias ? bg : nullptr;
    p.idx = idx; p.w = w; p.counts = counts; p.logits = logits;
    p.noise = noise;
    p.err = device_error_word();
    const bool dense = dense_routing(c);
    const int K = dense ? 0 : c.k;
    // Tiles of 128 tokens, one per CTA, while they fit on the SMs at once. 64-token tiles
    // (twice the CTAs, two per SM, half the ring each) measured slower: 21 against 20 us per
    // route call at 8192 tokens and 38 against 32 us at 16384 tokens and 128 experts. With
    // more tiles than SMs, top-k with k < 8 runs one CTA per SM over equal shares of tiles (the
    // tile shrinks so that every CTA takes the same number), and selects over one tile while
    // the next one loads.
    const int n_sm = num_sms();
    p.rows = RBM;
    int grid;
    if (K > 0 && K < 8 && c.T > RBM * n_sm) {
        const int per_cta = ceil_div(c.T, RBM * n_sm);
        p.rows = ceil_div(c.T, per_cta * n_sm);
        p.tiles = ceil_div(c.T, p.rows);
        grid = std::min(p.tiles, n_sm);
    } else {
        p.tiles = ceil_div(c.T, p.rows);
        grid = p.tiles;
    }
    CUtensorMap tx, tw;
    if (!make_map(&tx, x, (uint64_t)c.d, (uint64_t)c.T, (uint32_t)p.rows)) return cudaErrorInvalidValue;
    if (!make_map(&tw, Wg, (uint64_t)c.d, (uint64_t)c.E, (uint32_t)p.E_pad)) return cudaErrorInvalidValue;
    // shared memory: the ring, barriers, TMEM slot, counts and bias, and (k < 8) two buffers of
    // the groups' top-k lists (value and id per entry)
    const int G = route_groups(K, p.E_pad);
    const size_t fixed = 1024 + (2 * RMAX_STAGES + 8) * sizeof(uint64_t) + 16 + 2 * MOE_MAX_EXPERTS * sizeof(int);
    const size_t scratch = (K > 0 && K < 8) ? (size_t)2 * G * RBM * K * 8 : 0;
    const size_t ring_max = std::min<size_t>(RSMEM_BUDGET, 227 * 1024 - fixed - scratch);
    p.stages = std::max(2, std::min(RMAX_STAGES, (int)(ring_max / route_stage_bytes(p.E_pad))));
    const size_t smem = fixed + (size_t)p.stages * route_stage_bytes(p.E_pad) + scratch;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    // the top-8 path's staging (logits, group lists, values, slots, counts) lies over the ring
    const size_t top8_bytes = (size_t)RBM * 4 * ((size_t)c.E + 4 * 8 + 8 + 8 + 1);
    if (K == 8 && top8_bytes > (size_t)p.stages * route_stage_bytes(p.E_pad)) return cudaErrorInvalidValue;
    switch (K) {
        case 0: return launch_k<0>(p, tx, tw, smem, grid, s);
        case 1: return launch_k<1>(p, tx, tw, smem, grid, s);
        case 2: return launch_k<2>(p, tx, tw, smem, grid, s);
        case 3: return launch_k<3>(p, tx, tw, smem, grid, s);
        case 4: return launch_k<4>(p, tx, tw, smem, grid, s);
        case 5: return launch_k<5>(p, tx, tw, smem, grid, s);
        case 6: return launch_k<6>(p, tx, tw, smem, grid, s);
        case 7: return launch_k<7>(p, tx, tw, smem, grid, s);
        case 8: return launch_k<8>(p, tx, tw, smem, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
