// Internal interfaces between the translation units of the MoE library.
#pragma once

#include "common.cuh"

namespace moe {

// MOE_OK for a config that moe_config_init has filled, else the status every entry point
// returns for it (MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED).
moe_status_t config_status(const moe_config_t* cfg);

// k = E: dense soft routing (every expert on every token, slot j = expert j). The bucket
// layout is then closed-form and no sort runs.
inline bool dense_routing(const moe_config_t& c) { return c.k == c.E; }

// Epilogues of the grouped GEMMs over expert buckets (rows of one 128-row tile always belong
// to a single expert because buckets are padded to cfg.row_align rows, a multiple of 128).
enum GemmKind : int {
    kGemmFfn1 = 0,   // A = Xp W1_e^T + b1_e; store H = GELU(A) and Gp = GELU'(A)
    kGemmFfn2 = 1,   // Yp = H W2_e^T + b2_e
    kGemmDH = 2,     // dA = (dYp W2_e) * Gp
    kGemmDX = 3,     // dXp = dA W1_e
    kGemmWgrad = 4,  // dW_e = P_e^T Q_e over the rows of bucket e (dW2: P=dYp,Q=H; dW1: P=dA,Q=Xp)
    kGemmAccum = 5,  // out = aux + A B (in place on aux: dx += dz Wg of the soft balance loss)
    kGemmWgradF32 = 6,  // as kGemmWgrad with an fp32 output written from registers (split-K partials)
};

struct RowGemmArgs {
    int kind;
    const void* A;          // [rows, K] row-major activations
    const void* B;          // expert weights (layout per kind)
    const void* bias;       // [E, N] (Ffn1, Ffn2)
    const void* aux;        // [rows, N] Gp = GELU'(A) of the forward (DH)
    void* out0;             // [rows, N]
    void* out1;             // [rows, N] (H of Ffn1; out0 then holds Gp)
    const int32_t* offsets; // [E+1] bucket starts
    float* colsum;          // DH on tensor cores: column-sum partials of dA [tiles*4, N], or null
    int E, N, K;
    int rows_capacity;
    long long sBe, sBn, sBk; // element strides of B: expert, output column, reduction index
    int rows_valid = 0;      // rows of out0/aux that exist (0: rows_capacity); kGemmAccum
};

struct WgradArgs {
    const void* P;          // [rows, M] row-major
    const void* Q;          // [rows, N] row-major
    void* C;                // [E, M, N]
    const int32_t* offsets;
    int E, M, N;
    int rows_p = 0, rows_q = 0;   // rows of P and Q (0: cfg.rows_capacity)
    bool f32 = false;             // C is fp32 [E, M, N] (kGemmWgradF32)
    const int32_t* rows_used = nullptr;   // [E] rows of each bucket with an assignment (or null)
};

// router.cu
// noise: scratch [E, T] for the routing noise (needed when c.noise_std > 0 on the tensor-core
// path; drawn there once per call by a full-occupancy kernel)
cudaError_t launch_route(const moe_config_t& c, const void* x, const void* Wg, const float* bg,
                         int32_t* idx, float* w, int32_t* counts, float* balance_loss, float* logits,
                         float* noise, cudaStream_t s);

// router_tc.cu: gate GEMM on tcgen05 + top-k + softmax + counts (bf16, d % 64 == 0)
bool tc_route_supported(const moe_config_t& c);
cudaError_t launch_route_tc(const moe_config_t& c, const void* x, const void* Wg, const float* bg,
                            int32_t* idx, float* w, int32_t* counts, float* logits, const float* noise,
                            cudaStream_t s);

// dispatch.cu: stable counting sort of the assignments by expert
struct SortScratch {
    int32_t* blk_hist;     // [nblk, E] per-chunk expert histograms
    int32_t* assign_off;   // [E+1] exclusive scan of counts
    int32_t* assign_tok;   // [T*k] assignment (t*k+j) in expert-major, token-minor order
};
int sort_blocks(int T);
void sort_scratch_take(Workspace& ws, const moe_config_t& c, SortScratch* s);
// kept/offsets/row_token/slot_row/n_dropped may be null (assignment sort only).
cudaError_t launch_sort(const moe_config_t& c, const int32_t* idx, const SortScratch& s,
                        int32_t* kept, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                        int32_t* n_dropped, cudaStream_t st);
cudaError_t launch_dense_layout(const moe_config_t& c, const int32_t* idx, int32_t* kept, int32_t* offsets,
                                int32_t* row_token, int32_t* slot_row, int32_t* n_dropped, cudaStream_t st);
// used[e] = rows of bucket e that hold an assignment (row_token >= 0), from the bucket layout.
cudaError_t launch_bucket_used(const moe_config_t& c, const int32_t* offsets, const int32_t* row_token,
                               int32_t* used, cudaStream_t st);
cudaError_t launch_gather(const moe_config_t& c, const void* x, const int32_t* offsets,
                          const int32_t* row_token, const int32_t* slot_row, void* Xp, cudaStream_t st);

// gemm_simt.cu (fp32, and bf16 shapes the tensor-core kernel does not take)
cudaError_t launch_row_gemm_simt(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s);
cudaError_t launch_wgrad_simt(const moe_config_t& c, const WgradArgs& a, cudaStream_t s);

// gemm_tc.cu (bf16 on tcgen05 tensor cores; returns cudaErrorNotSupported for shapes it
// does not take)
bool tc_gemm_supported(const moe_config_t& c);
cudaError_t launch_row_gemm_tc(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s);
cudaError_t launch_wgrad_tc(const moe_config_t& c, const WgradArgs& a, cudaStream_t s);
// gemm_tc_pair.cu: weight gradients on CTA pairs (tcgen05.mma.cta_group::2, 256 x 256 tiles)
cudaError_t launch_wgrad_tc_pair(const moe_config_t& c, const WgradArgs& a, cudaStream_t s);
// row GEMMs on CTA pairs: 256-row tiles of each bucket (an odd bucket's last tile computes a
// second half past the bucket's end, not stored)
cudaError_t launch_row_gemm_tc_pair(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s);

// soft_balance.cu: differentiable balance loss on the soft load
struct SoftScratch {
    float* part;     // [chunks, E] per-chunk soft loads
    float* dz;       // [T, E] gradient of the logits
    float* dwg_part; // [splits, E, d]
    // tensor-core contractions (bf16, d % 64 == 0): dz split into bf16 hi and lo parts
    void* dzs;       // [T_pad, K2] bf16: columns [0,E) hi, [E8, E8+E) lo, zero elsewhere
    void* wge;       // [K2, d] bf16: Wg in rows [0,E) and [E8, E8+E), zero elsewhere
    int32_t* offs;   // [splits + 1] token buckets of the dz^T x split-K, then [0, T_pad]
    float* wpart;    // [splits, K2, d] fp32 split-K partials of dzs^T x
    float* dbg_part; // [blocks, E] partial column sums of dz
};
int soft_chunks(const moe_config_t& c);
int soft_splits(const moe_config_t& c);
void soft_scratch_take(Workspace& ws, const moe_config_t& c, SoftScratch* s);
cudaError_t launch_soft_balance(const moe_config_t& c, const float* logits, float weight, float* P,
                                float* loss, const SoftScratch& s, cudaStream_t st);
// dz^T x and dz Wg on tcgen05 (bf16 layers with d % 64 == 0 and E >= 32).
bool soft_tc_ok(const moe_config_t& c);

// dWg (+)= dz^T x and dbg (+)= column sums of dz for a dense dz [T, E] (split-K partials in
// s.dwg_part, fixed-order reductions); accumulate = false overwrites dWg and dbg.
cudaError_t launch_dense_dwg(const moe_config_t& c, const float* dz, const void* x, float* dWg, float* dbg,
                             bool accumulate, const SoftScratch& s, cudaStream_t st);
// win_n: null for one batch; for a window mean load P (moe_soft_balance_window), the device
// count of batches in the window (the gradient is divided by it and the mean taken from P).
cudaError_t launch_soft_balance_bwd(const moe_config_t& c, const float* logits, const float* P, float weight,
                                    const int32_t* win_n, const void* x, const void* Wg, void* dx, float* dWg,
                                    float* dbg, const SoftScratch& s, cudaStream_t st);
// Sliding window of soft loads: P (this batch) into ring slot state[0], Pbar = mean of the
// window's loads, loss on Pbar, state advanced.
cudaError_t launch_soft_window(const moe_config_t& c, const float* P, float weight, int W, float* ring,
                               int32_t* state, float* Pbar, float* loss, cudaStream_t st);

// coselect.cu: expert co-selection matrix H [E, E]
cudaError_t launch_coselect(const moe_config_t& c, const int32_t* idx, int32_t* H, cudaStream_t s);

// combine.cu
cudaError_t launch_combine(const moe_config_t& c, const void* Yp, const int32_t* slot_row,
                           const float* w, void* y, cudaStream_t s);
cudaError_t launch_combine_bwd(const moe_config_t& c, const void* dy, const void* Yp,
                               const float* w, const int32_t* offsets, const int32_t* row_token,
                               const int32_t* slot_row, void* dYp, float* dw, float* lossblk,
                               cudaStream_t s);
int combine_bwd_blocks(const moe_config_t& c);
// Router backward + un-permute (dz, dx). dz_dense (nullable; k <= MOE_MAX_K and E <= 32): also
// write dz as dense [T, E] rows. Block 0 also writes the reported loss when `loss` is set.
// dz_in: take dz from `dz` (written by launch_router_dz) and compute dx only.
cudaError_t launch_router_bwd(const moe_config_t& c, const float* w, const float* dw,
                              const int32_t* idx, const int32_t* slot_row, const void* Wg,
                              const void* dXp, float* dz, void* dx, float* dz_dense,
                              const float* lossblk, const float* balance_loss, float* loss, bool dz_in,
                              cudaStream_t s);
// The softmax Jacobian alone: dz [T, k], optionally dense [T, E] rows (k <= MOE_MAX_K), and
// (block 0) the reported loss.
cudaError_t launch_router_dz(const moe_config_t& c, const float* w, const float* dw, const int32_t* idx,
                             float* dz, float* dz_dense, const float* lossblk, const float* balance_loss,
                             float* loss, cudaStream_t s);
int dwg_chunks(const moe_config_t& c);
cudaError_t launch_dwg(const moe_config_t& c, const void* x, const float* dz,
                       const SortScratch& srt, float* part, float* dWg, float* dbg, cudaStream_t s);
// Bias gradients: column sums of a bucketed matrix. Partials hold one row per 32-row quarter
// of every 128-row tile: part [(rows_capacity / MOE_ROW_ALIGN) * 4, width] floats.
constexpr int kColsumParts = 4;
cudaError_t launch_colsum(const moe_config_t& c, const void* M, int width, const int32_t* offsets,
                          float* part, cudaStream_t s);
cudaError_t launch_bias_reduce(const moe_config_t& c, const float* part, int width,
                               const int32_t* offsets, float* db, cudaStream_t s);
cudaError_t launch_loss(const moe_config_t& c, const float* lossblk, const float* balance_loss,
                        float* loss, cudaStream_t s);

}  // namespace moe
