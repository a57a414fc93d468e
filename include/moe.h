/*
 * moe.h - C ABI of the GB300 (sm_103a) MoE layer library (libmoe.so): token routing and
 * expert compute, forward and backward, on one GPU.
 *
 * The layer (pages cited by title and section):
 *   z   = x Wg^T (+ bg)                                   gate linear
 *   idx = top-k of z per token (ties -> lower expert id)  top-k selection
 *   w   = softmax(z[idx] / temperature) over the k        routing weights
 *   k = E is dense soft routing (the naive soft MoE of the Expert-Parallelism page, section
 *   2.2: every expert runs on every token): nothing is selected, slot j holds expert j and
 *   w = softmax(z / temperature) over all E.
 *     "Native MoE training system PithTrain", section 4.1 (PithTrainMoELayer.forward:
 *     gate, torch.topk, softmax over the selected values); "Expert Parallelism: Scaling
 *     Mixture-of-Experts Models", section 2.2 (softmax(gate(x)/temperature); hybrid top-8
 *     pre-selection with soft weights over the 8), section 5.5 (route in FP32).
 *   counts[e], balance_loss = mean_e (counts[e] - mean(counts))^2
 *     "PyTorch distributed MoE training", section 3.3 (balance_loss).
 *   capacity C = ceil(capacity_factor * T * k / E); assignment (t,j) -> e is kept iff
 *   fewer than C earlier tokens picked e
 *     PithTrain page, section 4.3 item 1 (capacity, overflow tokens dropped).
 *   Xp = x rows permuted into expert buckets (token order inside a bucket)
 *     Expert-Parallelism page, section 4.2 idea 2 (tokens written straight into
 *     per-expert bucket offsets; one-device form of the sparse dispatch).
 *   per expert e: A = Xp_e W1_e^T + b1_e, H = GELU(A) (erf form), Yp = H W2_e^T + b2_e
 *     PyTorch-MoE page, section 3.2 (Expert); PithTrain page, section 4.1 (expert_pool).
 *   y[t] = sum over kept slots j of w[t,j] Yp[row(t,j)]
 *     PithTrain page, section 4.1 (output[mask] += expert_output * routing_weight).
 *   backward of L = sum(y * dy) (+ aux_loss_weight * balance_loss, which has no gradient)
 *     PithTrain page, section 4.2 (loss.backward()); PyTorch-MoE page, section 4.3
 *     (aux_loss_weight = 0.01).
 *
 * Conventions (every entry point):
 * - Pointers named as device pointers must point to device memory of the current device;
 *   host pointers are only the moe_config_t. The caller owns every buffer; the library
 *   allocates no device memory and keeps no per-call state. Outputs are overwritten.
 * - Activation, weight and scratch arrays (x, Wg, W1, b1, W2, b2, Xp, Gp, H, Yp, y, dy, dx,
 *   dW1, dW2 and ws) are read and written in 16-byte vectors and by TMA: their base
 *   addresses must be 16-byte aligned (cudaMalloc and PyTorch allocations are), else the
 *   call returns MOE_ERR_INVALID_ARG.
 * - All layouts are row-major, dense, following nn.Linear: x [T,d], Wg [E,d], bg [E] fp32,
 *   W1 [E,d_ff,d], b1 [E,d_ff], W2 [E,d,d_ff], b2 [E,d]. "act" below means the element
 *   type selected by cfg->dtype: fp32 (MOE_F32) or bf16 (MOE_BF16) for x, weights,
 *   activations and their gradients. Routing weights, logits and bias gradients are fp32.
 * - Permuted rows live in expert buckets: bucket e holds rows [offsets[e], offsets[e+1]),
 *   offsets[e] is a multiple of cfg->row_align (128 rows, set by moe_config_init), the
 *   first kept[e] rows are expert e's tokens in ascending token order and the rest of the
 *   bucket is padding (row_token = -1, zero rows in Xp). Buffers of permuted rows have
 *   cfg->rows_capacity rows.
 * - Calls are asynchronous on `stream` and never synchronise the host (except
 *   moe_get_error). Nothing that depends on data (counts, offsets) is read back.
 * - The library keeps a few per-device handles for the life of the process (its side stream,
 *   the device addresses of its error word and of the moe_dispatch_noalloc scratch array).
 *   cudaDeviceReset invalidates them: a process must not call the library on a device after
 *   resetting that device.
 * - Host-side validation failures return MOE_ERR_INVALID_ARG (bad value, null pointer) or
 *   MOE_ERR_UNSUPPORTED (valid but not implemented) and launch nothing. A failed launch
 *   returns MOE_ERR_CUDA. Faults detected on the device (a bounded wait that ran out, an
 *   index out of range) set a device error word that moe_get_error reports.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,
    MOE_ERR_UNSUPPORTED = -2,
    MOE_ERR_CUDA = -3,
    MOE_ERR_DEVICE_TIMEOUT = -4,
    MOE_ERR_DEVICE_BOUNDS = -5
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

#define MOE_ROW_ALIGN 128   /* bucket alignment (rows); cfg->row_align */
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_K 8           /* largest top-k selection; k = E (dense) is allowed for any E */

typedef struct {
    /* set by the caller */
    int32_t T;                 /* tokens, >= 0 */
    int32_t d;                 /* model dim, >= 1 */
    int32_t E;                 /* experts, 1..MOE_MAX_EXPERTS */
    int32_t k;                 /* experts per token: 1..min(E, MOE_MAX_K) (top-k), or E
                                  (dense soft routing, slot j = expert j) */
    int32_t d_ff;              /* expert hidden dim, >= 1 */
    float capacity_factor;     /* <= 0: no capacity limit */
    float temperature;         /* > 0: softmax(z_sel / temperature) */
    float aux_loss_weight;     /* weight of balance_loss in the reported loss (0.01 on the pages) */
    int32_t has_gate_bias;     /* 0/1: bg is added to the logits */
    int32_t dtype;             /* moe_dtype_t */
    float noise_std;           /* >= 0: training-time routing noise, logits += noise_std * N(0,1)
                                  before top-k and softmax ("PyTorch distributed MoE training",
                                  section 4.3: randn_like(logits) * 0.1); 0 = off */
    uint32_t noise_seed;       /* noise of experts 4g .. 4g+3 of token t: one Philox4x64-10
                                  draw at counter (t, g, 0, 0), key (noise_seed, 0); the top
                                  24 bits of outputs (0, 1) and (2, 3) give two pairs u1, u2 in
                                  (0,1], each turned into sqrt(-2 ln u1) cos(2 pi u2) and
                                  sqrt(-2 ln u1) sin(2 pi u2), in that order.
                                  Vary the seed from step to step. */
    /* derived by moe_config_init */
    int32_t capacity;          /* ceil(capacity_factor*T*k/E) in double, or INT32_MAX */
    int32_t rows_capacity;     /* rows of every permuted buffer (Xp, A, H, Yp) */
    int32_t row_align;         /* bucket alignment: MOE_ROW_ALIGN (128 rows). When the average
                                  bucket can reach 1024 rows (min(T*k, E*C)/E >= 1024) the
                                  expert GEMMs run 256-row tiles on CTA pairs (the last tile of
                                  a bucket with an odd number of 128-row tiles computes a second
                                  half it does not store); otherwise 128-row tiles on one CTA */
} moe_config_t;

/* Validates the caller's fields and fills the derived ones. Must be called before any
 * other entry point. Errors: MOE_ERR_INVALID_ARG (out-of-range field), MOE_ERR_UNSUPPORTED
 * (T*k or rows_capacity*max(d,d_ff) beyond 2^31-1). */
MOE_API moe_status_t moe_config_init(moe_config_t* cfg);

/* Bytes of device scratch (`ws`) the entry points need for this configuration; one buffer
 * of this size serves every call. Returns 0 for an invalid cfg. Aligned to 256 bytes. */
MOE_API size_t moe_workspace_bytes(const moe_config_t* cfg);

/* Gate linear + top-k + softmax over the k + expert counts + balance loss.
 *   x [T,d] act, Wg [E,d] act, bg [E] fp32 (read iff cfg->has_gate_bias, else may be NULL)
 *   -> idx [T,k] int32 (slot j = j-th largest logit; with k = E, slot j = expert j),
 *      w [T,k] fp32 (rows sum to 1), counts [E] int32 (pre-capacity choices, sum = T*k;
 *      T each with k = E), balance_loss [1] fp32,
 *      logits [T,E] fp32 (nullable: the routing logits z = x Wg^T + bg + noise; needed by
 *      moe_soft_balance).
 * Logits are accumulated in fp32. All pointers are device pointers. `ws` (moe_workspace_bytes)
 * holds the routing noise when cfg->noise_std > 0 (drawn once per call, then added to the
 * logits); it may be NULL when there is no noise. */
MOE_API moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wg, const float* bg,
                       int32_t* idx, float* w, int32_t* counts, float* balance_loss,
                       float* logits, void* ws, moe_stream_t stream);

/* Capacity, stable counting sort into expert buckets and the gather of x.
 *   idx [T,k] int32, x [T,d] act
 *   -> kept [E] int32 (= min(counts, capacity)), offsets [E+1] int32 (bucket starts,
 *      multiples of cfg->row_align, offsets[E] = rows in use), row_token [rows_capacity]
 *      int32 (token of each row; -1 on padding; rows >= offsets[E] unspecified),
 *      slot_row [T,k] int32 (row of assignment (t,j), -1 if dropped), n_dropped [1] int32,
 *      Xp [rows_capacity, d] act (rows >= offsets[E] unspecified).
 * Priority for capacity is token order. idx entries must lie in [0,E) and differ within a
 * token; a violation sets MOE_ERR_DEVICE_BOUNDS on the device. With k = E every bucket holds
 * tokens 0..min(T,C)-1 in order and idx must be the identity (idx[t,j] = j; else
 * MOE_ERR_DEVICE_BOUNDS); no sort runs. */
MOE_API moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* idx, const void* x,
                          int32_t* kept, int32_t* offsets, int32_t* row_token, int32_t* slot_row,
                          int32_t* n_dropped, void* Xp, void* ws, moe_stream_t stream);

/* moe_dispatch for callers that cannot allocate device memory. The pages have no
 * counterpart: this entry point exists for code that may not call cudaMalloc (it runs
 * inside a memory budget or a host framework that owns every allocation, or it is a plugin
 * given only its input and output buffers) and so cannot provide the `ws` scratch.
 * Same arguments, results and errors as moe_dispatch, minus `ws`: the sort scratch is a
 * fixed array of MOE_NOALLOC_SCRATCH_BYTES in the library's device memory, reserved on
 * every GPU that loads the library until the process exits. The call allocates nothing.
 * Limits: T <= MOE_NOALLOC_MAX_TOKENS and T*k <= MOE_NOALLOC_MAX_ASSIGNMENTS; larger
 * configurations return MOE_ERR_UNSUPPORTED (use moe_dispatch with a workspace). With
 * k = E (dense routing) no sort and no scratch are used and the limits do not apply.
 * Each call looks up the array's device address (a host lookup; the first one on a device
 * may load the library's device code, so make a first call before any stream capture, as
 * for every entry point). All calls share the one array: calls that
 * may overlap on the GPU (other streams, other host threads) race and must be serialised
 * by the caller. Nothing in the array needs to start at zero; each call writes what it
 * reads. */
#define MOE_NOALLOC_SCRATCH_BYTES (2u << 20)
#define MOE_NOALLOC_MAX_TOKENS 65536
#define MOE_NOALLOC_MAX_ASSIGNMENTS 262144
MOE_API moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const int32_t* idx, const void* x,
                                          int32_t* kept, int32_t* offsets, int32_t* row_token,
                                          int32_t* slot_row, int32_t* n_dropped, void* Xp,
                                          moe_stream_t stream);

/* Per-expert FFN over the buckets: A = Xp W1_e^T + b1_e, H = GELU(A), Yp = H W2_e^T + b2_e.
 *   Xp [rows_capacity,d], offsets [E+1] (from moe_dispatch), W1 [E,d_ff,d], b1 [E,d_ff],
 *   W2 [E,d,d_ff], b2 [E,d] -> Gp, H [rows_capacity,d_ff], Yp [rows_capacity,d] (all act;
 *   rows >= offsets[E] untouched). Gp = GELU'(A) = Phi(A) + A phi(A) is what the backward
 *   needs of the pre-activation, saved in place of A itself. fp32 accumulation. */
MOE_API moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* Xp, const int32_t* offsets,
                            const void* W1, const void* b1, const void* W2, const void* b2,
                            void* Gp, void* H, void* Yp, void* ws, moe_stream_t stream);

/* Weighted combine back to token order: y[t] = sum_{j: slot_row[t,j] >= 0} w[t,j] Yp[slot_row[t,j]],
 * accumulated in fp32; a token whose slots were all dropped gets 0.  y [T,d] act. */
MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const void* Yp, const int32_t* slot_row,
                         const float* w, void* y, moe_stream_t stream);

/* Backward of the layer for the gradient seed dy [T,d] act, from the forward's saved tensors.
 *   inputs : dy, x, Wg, idx, w, offsets, row_token, slot_row, Xp, Gp, H, Yp, W1, W2 (as above),
 *            balance_loss [1] (nullable; enters the reported loss only)
 *   outputs: dx [T,d] act, dWg [E,d] fp32, dW1 [E,d_ff,d] act, db1 [E,d_ff] fp32,
 *            dW2 [E,d,d_ff] act, db2 [E,d] fp32, dbg [E] fp32 (nullable: gate-bias
 *            gradient, written only when cfg->has_gate_bias), dw [T,k] fp32 (nullable:
 *            gradient of the routing weights),
 *            loss [1] fp32 (nullable: sum(y*dy) + aux_loss_weight*balance_loss).
 * Dropped assignments give dw = 0 but still enter their token's softmax Jacobian. Experts
 * with no kept rows get zero weight and bias gradients. Scratch comes from ws. Part of the
 * work runs on a side stream of the library that forks from and joins back into `stream`
 * (event waits, also valid while `stream` is being captured into a CUDA graph). */
MOE_API moe_status_t moe_backward(const moe_config_t* cfg, const void* dy, const void* x, const void* Wg,
                          const int32_t* idx, const float* w, const int32_t* offsets,
                          const int32_t* row_token, const int32_t* slot_row, const void* Xp,
                          const void* Gp, const void* H, const void* Yp, const void* W1,
                          const void* W2, const float* balance_loss,
                          void* dx, float* dWg, void* dW1, float* db1, void* dW2, float* db2,
                          float* dbg, float* dw, float* loss, void* ws, moe_stream_t stream);

/* Differentiable balance loss on the soft expert load. The integer counts of balance_loss
 * ("PyTorch distributed MoE training", section 3.3) have no gradient; here the same
 * squared-deviation form is applied to the soft load of the gate probabilities
 * ("Expert Parallelism: Scaling Mixture-of-Experts Models", sections 2.2-2.3):
 *   P_e = sum_t softmax(logits_t / temperature)_e,  loss = weight * mean_e (P_e - T/E)^2.
 *   logits [T,E] fp32 (from moe_route) -> P [E] fp32, loss [1] fp32. Fixed-order sums.
 * Scratch from ws (moe_workspace_bytes covers it). */
MOE_API moe_status_t moe_soft_balance(const moe_config_t* cfg, const float* logits, float weight,
                                      float* P, float* loss, void* ws, moe_stream_t stream);

/* Gradient of moe_soft_balance's loss, ADDED to the layer gradients:
 *   dz_te = p_te (g_e - sum_j p_tj g_j) / temperature, g_e = weight * 2 (P_e - T/E) / E,
 *   dx += dz Wg, dWg += dz^T x, dbg += sum_t dz (dbg nullable).
 *   logits [T,E], P [E] (from moe_soft_balance), x [T,d] act, Wg [E,d] act;
 *   dx [T,d] act, dWg [E,d] fp32, dbg [E] fp32 are read and updated in place. */
MOE_API moe_status_t moe_soft_balance_backward(const moe_config_t* cfg, const float* logits,
                                               const float* P, float weight, const void* x,
                                               const void* Wg, void* dx, float* dWg, float* dbg,
                                               void* ws, moe_stream_t stream);

/* The soft balance loss on a sliding window of batches: "Expert Parallelism: Scaling
 * Mixture-of-Experts Models", section 2.3 (the per-expert load is averaged over the last 100
 * batches before the balance loss is taken, because a single batch's load is too noisy).
 * The caller owns the window's state; the library keeps none:
 *   ring  [W, E] fp32 device: the soft loads of the last W batches (contents need no
 *         initialisation: only slots written by earlier calls are read)
 *   state [2] int32 device: state[0] = ring slot of the next batch, state[1] = batches in the
 *         window (0..W). Set both to 0 before the first call; a state out of range sets
 *         MOE_ERR_DEVICE_BOUNDS and the window restarts.
 * Each call computes this batch's soft load P_e = sum_t softmax(logits_t / temperature)_e
 * (as moe_soft_balance), stores it in slot state[0], and with n = min(state[1] + 1, W):
 *   Pbar [E] = mean of the n most recent soft loads (this batch included),
 *   loss [1] = weight * mean_e (Pbar_e - mean(Pbar))^2   (loss nullable),
 * then advances the state: state[0] = (state[0] + 1) mod W, state[1] = n.
 * W = 1 is moe_soft_balance. logits [T,E] fp32; P, Pbar [E] fp32 device; W in
 * 1..MOE_MAX_WINDOW; ring and state 4-byte aligned. Scratch from ws (moe_workspace_bytes).
 * Successive calls on one ring must be ordered on the GPU (one stream). */
#define MOE_MAX_WINDOW 4096
MOE_API moe_status_t moe_soft_balance_window(const moe_config_t* cfg, const float* logits, float weight,
                                             int32_t W, float* ring, int32_t* state, float* P, float* Pbar,
                                             float* loss, void* ws, moe_stream_t stream);

/* Gradient of moe_soft_balance_window's loss, ADDED to the layer gradients. The earlier
 * batches of the window are stored statistics, so the gradient reaches only this batch:
 *   g_e = weight * 2 (Pbar_e - mean(Pbar)) / (E n),  n = state[1],
 *   dz_te = p_te (g_e - sum_j p_tj g_j) / temperature,  dx += dz Wg, dWg += dz^T x,
 *   dbg += sum_t dz (dbg nullable).
 * Call it after the forward call of the same batch (which set state[1] = n) and before the
 * next one, with that call's Pbar and state. logits, x [T,d] act, Wg [E,d] act; dx, dWg, dbg
 * are read and updated in place. */
MOE_API moe_status_t moe_soft_balance_window_backward(const moe_config_t* cfg, const float* logits,
                                                      const float* Pbar, float weight, const int32_t* state,
                                                      const void* x, const void* Wg, void* dx, float* dWg,
                                                      float* dbg, void* ws, moe_stream_t stream);

/* Expert co-selection matrix of a batch: "Expert Parallelism: Scaling Mixture-of-Experts
 * Models", section 3.2, step 1 (experts chosen by the same token; the input of the page's
 * affinity-aware placement). The page calls the matrix asymmetric; accordingly, for i != j,
 *   H[i][j] = number of tokens whose top-k holds i in an earlier slot (higher logit) than j,
 * so H + H^T is the co-occurrence count, and H[i][i] = number of tokens that chose i.
 *   idx [T,k] int32 (as from moe_route) -> H [E,E] int32 (overwritten). Device pointers.
 * Entries out of [0,E) or repeated within a token set MOE_ERR_DEVICE_BOUNDS and are skipped.
 * With k = E > MOE_MAX_K (dense routing) idx must be the identity: H[i][j] = T for i <= j,
 * 0 below the diagonal; a token whose row is not the identity sets MOE_ERR_DEVICE_BOUNDS and
 * is not counted. */
MOE_API moe_status_t moe_coselect(const moe_config_t* cfg, const int32_t* idx, int32_t* H,
                                  moe_stream_t stream);

/* Synchronises `stream`, then returns and clears the device error word of the current
 * device: MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_BOUNDS; MOE_ERR_CUDA if the
 * stream reports a CUDA error. */
MOE_API moe_status_t moe_get_error(moe_stream_t stream);

/* Self-test of the device-side bounded waits (failure detection without a GPU fault). A
 * kernel waits on an object that nothing signals, through the wait helper the layer's kernels
 * use: an mbarrier phase wait, as in the tensor-core pipelines (mode 0, the only mode). After
 * budget_cycles (1e3 .. 4e9 SM clock cycles) the wait gives up, records
 * MOE_ERR_DEVICE_TIMEOUT in the device error word and the kernel returns; the context stays
 * usable.
 *   timed_out: device int32, set to the number of waits that ran out (1)
 *   scratch  : unused (may be null)
 * Returns MOE_ERR_INVALID_ARG for a mode other than 0, a bad budget or a null timed_out; the
 * timeout itself is read with moe_get_error. */
MOE_API moe_status_t moe_selftest_wait_timeout(int32_t mode, int64_t budget_cycles, int32_t* timed_out,
                                               void* scratch, moe_stream_t stream);

/* Kernel trace: the device time of every kernel the library launches, for profiling from
 * the host without an external profiler. The pages have no counterpart.
 * moe_trace_begin opens a trace on the calling host thread, with room for max_launches
 * (1 .. 65536) launches; it creates 2 * max_launches CUDA timing events (no device memory)
 * and discards the previous trace's results. Until moe_trace_end, every kernel the library
 * launches from this thread, on a stream that is not being captured into a graph, is
 * bracketed by two events recorded on its own stream: the kernel then starts only after the
 * previous work of its stream has finished (no overlap with a dependent launch), so each
 * duration is the kernel's own; while a trace is open, moe_backward also keeps its two
 * branches from overlapping (its caller's stream waits for the side branch). Launches beyond
 * max_launches are not traced (counted by moe_trace_dropped).
 * moe_trace_end synchronises the recorded events and returns the number of traced launches
 * (>= 0), or MOE_ERR_INVALID_ARG if no trace is open, or MOE_ERR_CUDA.
 * moe_trace_record gives launch i's kernel name (without parameters, e.g.
 * "route_tc_kernel<2>"; the string stays valid until the next moe_trace_begin on this thread)
 * and its duration in milliseconds, in launch order. */
MOE_API moe_status_t moe_trace_begin(int32_t max_launches);
MOE_API int32_t moe_trace_end(void);
MOE_API moe_status_t moe_trace_record(int32_t i, const char** name, float* ms);
MOE_API int32_t moe_trace_dropped(void);

/* Static description of a status code (never NULL). */
MOE_API const char* moe_status_str(moe_status_t status);

/* Number of kernels this library has launched in this process (all devices). */
MOE_API uint64_t moe_kernel_launches(void);

/* Library version string, e.g. "moe-gb300 0.1 sm_103a". */
MOE_API const char* moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
