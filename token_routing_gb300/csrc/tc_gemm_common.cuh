// Pieces shared by the tcgen05 grouped-GEMM kernels (one-CTA and CTA-pair variants): tile
// geometry, kernel parameters, bucket lookup, and the epilogue's staging / TMA-store helpers.
#pragma once

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
// Epilogue staging: per epilogue warp two 2 KB buffers of 32 rows x 64 bytes (64-byte
// swizzle) from which TMA stores write coalesced 32x32 bf16 boxes.
constexpr int STG_BYTES = 2048;
constexpr int EPI_SMEM = EPI_WARPS * 2 * STG_BYTES;

struct TcParams {
    int kind;                 // GemmKind
    const int32_t* offsets;   // [E+1] bucket starts
    int E, N, K, M;           // row GEMMs: out [rows, N], K reduction (kGemmAccum: M = rows that
                              // exist in aux/out); wgrad: C_e [M, N]
    int n_tiles, m_tiles;
    const __nv_bfloat16* bias;   // [E, N]
    const __nv_bfloat16* aux;    // [rows, N] (A of the forward, for dH)
    __nv_bfloat16* out0;
    __nv_bfloat16* out1;
    float* outf;                 // kGemmWgradF32: fp32 [E, M, N]
    float* colsum;               // dH: per-(tile, lane quarter) column sums of dA, or null
    const int32_t* rows_used;    // wgrad (bf16): rows of bucket e that hold assignments, or null
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

// Pair tiles of the row GEMMs on CTA pairs: bucket e (128-row aligned, n_e tiles of 128 rows)
// has ceil(n_e / 2) pair tiles of 256 rows; when n_e is odd the last one's second half lies
// past the bucket's end (its rows are computed but not stored). s_q[e] = number of buckets
// before e with an odd n_e (<= 256, so 16 bits), s_q[E] = all of them; the pair tiles before
// bucket e then number (offsets[e] / 128 + s_q[e]) / 2. Warp 0 only (E <= 256: 8 buckets per
// lane, then a warp scan of the lane sums).
__device__ __forceinline__ void bucket_odd_prefix(const int* s_off, int E, uint16_t* s_q, int lane) {
    int odd[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        odd[i] = e < E ? (((s_off[e + 1] - s_off[e]) / BM) & 1) : 0;
        sum += odd[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane * 8 + i;
        if (e < E) s_q[e] = (uint16_t)run;
        run += odd[i];
    }
    if (lane == 31) s_q[E] = (uint16_t)incl;
}

// Number of pair tiles in buckets 0 .. e-1.
__device__ __forceinline__ int pairs_before(const int* s_off, const uint16_t* s_q, int e) {
    return (s_off[e] / BM + (int)s_q[e]) >> 1;
}

// The bucket of pair tile r: the largest e with pairs_before(e) <= r.
__device__ __forceinline__ int bucket_of_pair(const int* s_off, const uint16_t* s_q, int E, int r) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pairs_before(s_off, s_q, mid) <= r) lo = mid; else hi = mid - 1;
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

// 32 bf16 (64 bytes) as raw vectors: fetched one chunk ahead of their use.
struct Raw32 {
    uint4 q[4];
};
__device__ __forceinline__ void load_raw32(Raw32& r, const __nv_bfloat16* src) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r.q[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
}
__device__ __forceinline__ void unpack_raw32(const Raw32& r, float* out) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.q[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            out[8 * i + 2 * j] = f.x;
            out[8 * i + 2 * j + 1] = f.y;
        }
    }
}

template <int KIND>
constexpr bool has_bias() { return KIND == kGemmFfn1 || KIND == kGemmFfn2; }

// The side input (aux [rows, N] bf16) of one 32-row x 32-column chunk, read coalesced: lane l
// loads the 16-byte segment l & 3 of rows aux_row0 + 8 i (aux_row0 = the warp's first row +
// (l >> 2)). kGemmAccum reads zeros for rows at or beyond p.M (rows that do not exist).
template <int KIND>
__device__ __forceinline__ void load_aux32(Raw32& r, const TcParams& p, size_t aux_row0, int n, int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const size_t row = aux_row0 + 8 * i;
        if (KIND == kGemmAccum && row >= (size_t)p.M) r.q[i] = make_uint4(0u, 0u, 0u, 0u);
        else r.q[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + row * p.N + n + (lane & 3) * 8));
    }
}

__device__ __forceinline__ uint32_t sw64_addr(uint32_t base, int row, int j) {
    return base + row * 64 + ((j ^ ((row >> 1) & 3)) << 4);
}
__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint4 pack8(const float* v) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return u;
}
__device__ __forceinline__ void unpack8(const uint4& u, float* out) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(src) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// One epilogue warp's staging buffers and store count (buffer = count & 1).
struct Stager {
    uint32_t base;
    int count;
    // Returns the next buffer once the TMA store that last read it has finished.
    __device__ __forceinline__ uint32_t acquire(int lane) {
        if (lane == 0 && count >= 2) bulk_wait_read1();
        __syncwarp();
        return base + (count & 1) * STG_BYTES;
    }
    // Writes the lane's row (32 values) into `buf`, then one TMA store of the 32x32 box.
    __device__ __forceinline__ void store(int lane, uint32_t buf, const float* v, const CUtensorMap* tm, int x, int y) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sts128(sw64_addr(buf, lane, j), pack8(v + 8 * j));
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm, buf, x, y);
            bulk_commit();
        }
        ++count;
    }
    // Zeros to `boxes` 32x32 boxes side by side (columns x0, x0 + 32, ...; rows y .. y + 31)
    // from one zeroed buffer, in one bulk group: the weight-gradient tile of an expert that
    // received no rows.
    __device__ __forceinline__ void store_zero(int lane, uint32_t buf, const CUtensorMap* tm, int x0, int boxes, int y) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) sts128(buf + lane * 64 + j * 16, z);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            for (int i = 0; i < boxes; ++i) tma_store_2d(tm, buf, x0 + 32 * i, y);
            bulk_commit();
        }
        ++count;
    }
};

// Two outputs per 32-column chunk (Ffn1: GELU'(A) and H): NB buffer pairs of one epilogue
// warp (pair count % NB), one proxy fence and one bulk group per chunk.
template <int NB>
struct Stager2 {
    uint32_t base;
    int count;
    // Returns the next buffer pair once the TMA stores that last read it have finished.
    __device__ __forceinline__ uint32_t acquire(int lane) {
        if (lane == 0 && count >= NB) {
            if (NB == 1) bulk_wait_read0();
            else bulk_wait_read1();
        }
        __syncwarp();
        return base + (count % NB) * 2 * STG_BYTES;
    }
    // a: the lane's 32 biased pre-activations. Eight at a time: GELU'(a) into the first
    // buffer (tm0), GELU(a) into the second (tm1); then one fence and the two TMA stores.
    __device__ __forceinline__ void store_gelu(int lane, uint32_t buf, const float* a,
                                               const CUtensorMap* tm0, const CUtensorMap* tm1, int x, int y) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float g[8], gp[8];
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                gelu_and_grad_f2(a[8 * j + i], a[8 * j + i + 1], g[i], g[i + 1], gp[i], gp[i + 1]);
            sts128(sw64_addr(buf, lane, j), pack8(gp));
            sts128(sw64_addr(buf + STG_BYTES, lane, j), pack8(g));
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm0, buf, x, y);
            tma_store_2d(tm1, buf + STG_BYTES, x, y);
            bulk_commit();
        }
        ++count;
    }
};

// Column sums of the 32 x 32 bf16 chunk a Stager has just written to `buf` (lane = row,
// swizzled 64-byte rows), i.e. of the values the chunk stores. Lanes 0-15 add the even rows and
// lanes 16-31 the odd rows, each lane two adjacent columns read as one 32-bit word: a step reads
// one 128-byte line, with no bank conflicts. The two halves then combine across lanes l, l + 16.
// Lane l < 16 returns the sums of columns 2l and 2l + 1.
__device__ __forceinline__ float2 staged_colsum32(uint32_t buf, int lane) {
    const int c = lane & 15;
    const uint32_t off = (uint32_t)(c & 3) * 4;
    uint64_t acc = pk2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 2 * i + (lane >> 4);
        uint32_t w;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(sw64_addr(buf, r, c >> 2) + off));
        acc = add2(acc, pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)));
    }
    float s0, s1;
    upk2(acc, s0, s1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    return make_float2(s0, s1);
}

}  // namespace
}  // namespace moe
