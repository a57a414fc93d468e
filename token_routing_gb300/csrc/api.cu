// C ABI of the MoE layer library: argument validation, workspace layout and the order of
// kernel launches for each entry point. The arithmetic lives in router_tc.cu / router.cu,
// dispatch.cu, gemm_tc_pair.cu / gemm_tc.cu / gemm_simt.cu, combine.cu, soft_balance.cu and
// coselect.cu.
#include <climits>
#include <cmath>
#include <initializer_list>
#include <mutex>

#include "internal.cuh"

namespace moe {

std::atomic<uint64_t> g_launches{0};

namespace {

__device__ int g_err_word;  // one device error word per device (kErrNone / kErrTimeout / kErrBounds)

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return dev;
}

int64_t derived_capacity(const moe_config_t& c) {
    if (!(c.capacity_factor > 0.0f)) return INT32_MAX;
    const double cap = std::ceil((double)c.capacity_factor * (double)c.T * (double)c.k / (double)c.E);
    return cap > (double)INT32_MAX ? INT32_MAX : (int64_t)cap;
}

int64_t derived_nmax(const moe_config_t& c, int64_t cap) {
    return std::min((int64_t)c.T * c.k, (int64_t)c.E * cap);
}

// Buckets are padded to 128 rows (MOE_ROW_ALIGN), the row tile of the GEMMs.
int32_t derived_align(const moe_config_t&, int64_t) { return MOE_ROW_ALIGN; }

// The row GEMMs run on CTA pairs (256-row tiles; an odd bucket's last tile has a second half
// past the bucket's end that is computed but not stored) when an average bucket can reach 1024
// rows; below that most buckets are a few 128-row tiles and the one-CTA kernel takes them.
bool pair_rows(const moe_config_t& c) { return derived_nmax(c, derived_capacity(c)) >= 1024LL * c.E; }

int64_t derived_rows(const moe_config_t& c, int64_t cap) {
    const int64_t n_max = derived_nmax(c, cap);
    const int64_t align = derived_align(c, cap);
    const int64_t buckets = std::min<int64_t>(c.E, n_max);
    const int64_t rows = n_max + (align - 1) * buckets;
    return (rows + align - 1) / align * align;
}

moe_status_t check_fields(const moe_config_t* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d < 1 || c->E < 1 || c->E > MOE_MAX_EXPERTS || c->k < 1 ||
        (c->k > MOE_MAX_K && c->k != c->E) || c->k > c->E || c->d_ff < 1)
        return MOE_ERR_INVALID_ARG;
    if (!(c->temperature > 0.0f) || !std::isfinite(c->temperature)) return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(c->capacity_factor) || !std::isfinite(c->aux_loss_weight)) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->has_gate_bias != 0 && c->has_gate_bias != 1) return MOE_ERR_INVALID_ARG;
    if (!(c->noise_std >= 0.0f) || !std::isfinite(c->noise_std)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->T * c->k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    const int64_t rows = derived_rows(*c, derived_capacity(*c));
    if (rows > INT32_MAX || rows * (int64_t)std::max(c->d, c->d_ff) > ((int64_t)1 << 40))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// The entry points accept only a config that moe_config_init has filled.
moe_status_t check_config(const moe_config_t* c) {
    moe_status_t st = check_fields(c);
    if (st != MOE_OK) return st;
    const int64_t cap = derived_capacity(*c);
    if (c->capacity != cap || c->rows_capacity != derived_rows(*c, cap) || c->row_align != derived_align(*c, cap))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Activation, weight and scratch arrays are read and written in 16-byte vectors and by TMA:
// their base addresses must be 16-byte aligned (null pointers pass; they are checked apart).
bool aligned16(std::initializer_list<const void*> ps) {
    for (const void* p : ps)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return false;
    return true;
}

#define MOE_TRY(expr)                                   \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return MOE_ERR_CUDA;     \
    } while (0)

struct BackwardScratch {
    SortScratch sort;
    void* dYp;
    void* dA;
    void* dXp;
    float* dw;
    float* dz;
    float* lossblk;
    float* dwg_part;
    float* colsum_d;    // column-sum partials of dYp (db2)
    float* colsum_f;    // column-sum partials of dA (db1)
    SoftScratch soft;   // soft balance loss
    float* noise;       // routing noise [E, T] (expert-major), when cfg.noise_std > 0
    int32_t* used;      // [E] rows of each bucket holding an assignment (weight-gradient K)
};

size_t carve_backward(const moe_config_t& c, void* base, BackwardScratch* b) {
    Workspace ws{static_cast<char*>(base), 0};
    const size_t es = c.dtype == MOE_BF16 ? 2 : 4;
    const size_t R = (size_t)c.rows_capacity;
    sort_scratch_take(ws, c, &b->sort);
    b->dYp = ws.take<char>(R * c.d * es);
    b->dA = ws.take<char>(R * c.d_ff * es);
    b->dXp = ws.take<char>(R * c.d * es);
    b->dw = ws.take<float>((size_t)c.T * c.k + 1);
    b->dz = ws.take<float>((size_t)c.T * c.k + 1);
    b->lossblk = ws.take<float>((size_t)combine_bwd_blocks(c) + 1);
    b->dwg_part = ws.take<float>((size_t)c.E * dwg_chunks(c) * c.d);
    b->colsum_d = ws.take<float>((R / MOE_ROW_ALIGN) * kColsumParts * (size_t)c.d + 1);
    b->colsum_f = ws.take<float>((R / MOE_ROW_ALIGN) * kColsumParts * (size_t)c.d_ff + 1);
    b->noise = ws.take<float>(c.noise_std > 0.f ? (size_t)c.T * c.E + 1 : 1);
    b->used = ws.take<int32_t>((size_t)c.E + 1);
    soft_scratch_take(ws, c, &b->soft);
    return align_up(ws.used, 256);
}

// One non-blocking side stream per device for the backward's parallel branch (created on
// first use, kept until exit).
cudaStream_t g_side[kMaxDevices] = {};
cudaStream_t side_stream() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_side[dev]) {
        cudaStream_t st = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        g_side[dev] = st;
    }
    return g_side[dev];
}

// Fork/join events of one call; destroyed when the call returns (pending waits still hold).
struct EventSet {
    cudaEvent_t a = nullptr, b = nullptr, c = nullptr, d = nullptr, e = nullptr, f = nullptr;
    bool ok = false;
    explicit EventSet(bool extra) {
        ok = cudaEventCreateWithFlags(&a, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&b, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&c, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&d, cudaEventDisableTiming) == cudaSuccess &&
             (!extra || (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess &&
                         cudaEventCreateWithFlags(&f, cudaEventDisableTiming) == cudaSuccess));
    }
    ~EventSet() {
        for (cudaEvent_t x : {a, b, c, d, e, f})
            if (x) cudaEventDestroy(x);
    }
};

bool use_tc(const moe_config_t& c) { return c.dtype == MOE_BF16 && tc_gemm_supported(c); }

cudaError_t row_gemm(const moe_config_t& c, const RowGemmArgs& a, cudaStream_t s) {
    if (!use_tc(c)) return launch_row_gemm_simt(c, a, s);
    return pair_rows(c) ? launch_row_gemm_tc_pair(c, a, s) : launch_row_gemm_tc(c, a, s);
}
cudaError_t wgrad(const moe_config_t& c, const WgradArgs& a, cudaStream_t s) {
    if (c.rows_capacity == 0) {
        // no expert rows at all (an empty batch): every weight gradient is zero, and no
        // operand is touched
        const long long n = (long long)a.E * a.M * a.N;
        if (a.f32 || c.dtype != MOE_BF16) return launch_fill(static_cast<float*>(a.C), n, 0.f, s);
        return launch_fill(static_cast<uint16_t*>(a.C), n, (uint16_t)0, s);   // bf16 +0.0
    }
    return use_tc(c) ? launch_wgrad_tc_pair(c, a, s) : launch_wgrad_simt(c, a, s);
}

}  // namespace

moe_status_t config_status(const moe_config_t* cfg) { return check_config(cfg); }

int* device_error_word() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

int num_sms() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_num_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_config_init(moe_config_t* cfg) {
    moe_status_t st = check_fields(cfg);
    if (st != MOE_OK) return st;
    const int64_t cap = derived_capacity(*cfg);
    cfg->capacity = (int32_t)cap;
    cfg->rows_capacity = (int32_t)derived_rows(*cfg, cap);
    cfg->row_align = derived_align(*cfg, cap);
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_config_t* cfg) {
    if (check_config(cfg) != MOE_OK) return 0;
    BackwardScratch b;
    return carve_backward(*cfg, nullptr, &b);
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wg, const float* bg,
                       int32_t* idx, float* w, int32_t* counts, float* balance_loss, float* logits,
                       void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!Wg || !counts || !balance_loss || (cfg->has_gate_bias && !bg)) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!x || !idx || !w)) return MOE_ERR_INVALID_ARG;
    if (cfg->noise_std > 0.f && cfg->T > 0 && !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16({x, Wg, ws})) return MOE_ERR_INVALID_ARG;
    float* noise = nullptr;
    if (ws) {
        BackwardScratch b;
        carve_backward(*cfg, ws, &b);
        noise = b.noise;
    }
    return cuda_status(launch_route(*cfg, x, Wg, bg, idx, w, counts, balance_loss, logits, noise,
                                    (cudaStream_t)stream));
}

moe_status_t moe_soft_balance(const moe_config_t* cfg, const float* logits, float weight, float* P,
                              float* loss, void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!P || !ws || (cfg->T > 0 && !logits) || !std::isfinite(weight)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({ws})) return MOE_ERR_INVALID_ARG;
    BackwardScratch b;
    carve_backward(*cfg, ws, &b);
    return cuda_status(launch_soft_balance(*cfg, logits, weight, P, loss, b.soft, (cudaStream_t)stream));
}

moe_status_t moe_soft_balance_backward(const moe_config_t* cfg, const float* logits, const float* P,
                                       float weight, const void* x, const void* Wg, void* dx, float* dWg,
                                       float* dbg, void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!P || !Wg || !dWg || !ws || !std::isfinite(weight)) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!logits || !x || !dx)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({x, Wg, dx, ws})) return MOE_ERR_INVALID_ARG;
    BackwardScratch b;
    carve_backward(*cfg, ws, &b);
    return cuda_status(launch_soft_balance_bwd(*cfg, logits, P, weight, nullptr, x, Wg, dx, dWg, dbg, b.soft,
                                               (cudaStream_t)stream));
}

moe_status_t moe_soft_balance_window(const moe_config_t* cfg, const float* logits, float weight, int32_t W,
                                     float* ring, int32_t* state, float* P, float* Pbar, float* loss, void* ws,
                                     moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (W < 1 || W > MOE_MAX_WINDOW || !ring || !state || !P || !Pbar || !ws || (cfg->T > 0 && !logits) ||
        !std::isfinite(weight))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16({ws}) || (reinterpret_cast<uintptr_t>(ring) & 3u) || (reinterpret_cast<uintptr_t>(state) & 3u))
        return MOE_ERR_INVALID_ARG;
    BackwardScratch b;
    carve_backward(*cfg, ws, &b);
    cudaStream_t s = (cudaStream_t)stream;
    MOE_TRY(launch_soft_balance(*cfg, logits, weight, P, nullptr, b.soft, s));
    MOE_TRY(launch_soft_window(*cfg, P, weight, W, ring, state, Pbar, loss, s));
    return MOE_OK;
}

moe_status_t moe_soft_balance_window_backward(const moe_config_t* cfg, const float* logits, const float* Pbar,
                                              float weight, const int32_t* state, const void* x, const void* Wg,
                                              void* dx, float* dWg, float* dbg, void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!Pbar || !state || !Wg || !dWg || !ws || !std::isfinite(weight)) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!logits || !x || !dx)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({x, Wg, dx, ws}) || (reinterpret_cast<uintptr_t>(state) & 3u)) return MOE_ERR_INVALID_ARG;
    BackwardScratch b;
    carve_backward(*cfg, ws, &b);
    // state[1] is the window's batch count once the forward of this batch has run
    return cuda_status(launch_soft_balance_bwd(*cfg, logits, Pbar, weight, state + 1, x, Wg, dx, dWg, dbg, b.soft,
                                               (cudaStream_t)stream));
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* idx, const void* x, int32_t* kept,
                          int32_t* offsets, int32_t* row_token, int32_t* slot_row, int32_t* n_dropped,
                          void* Xp, void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!kept || !offsets || !n_dropped || !ws) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!idx || !x || !slot_row)) return MOE_ERR_INVALID_ARG;
    if (cfg->rows_capacity > 0 && (!row_token || !Xp)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({x, Xp, ws})) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (dense_routing(*cfg)) {
        MOE_TRY(launch_dense_layout(*cfg, idx, kept, offsets, row_token, slot_row, n_dropped, s));
    } else {
        Workspace w{static_cast<char*>(ws), 0};
        SortScratch srt;
        sort_scratch_take(w, *cfg, &srt);
        MOE_TRY(launch_sort(*cfg, idx, srt, kept, offsets, row_token, slot_row, n_dropped, s));
    }
    MOE_TRY(launch_gather(*cfg, x, offsets, row_token, slot_row, Xp, s));
    return MOE_OK;
}

moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* Xp, const int32_t* offsets,
                            const void* W1, const void* b1, const void* W2, const void* b2, void* Gp,
                            void* H, void* Yp, void* ws, moe_stream_t stream) {
    (void)ws;
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!offsets || !W1 || !b1 || !W2 || !b2) return MOE_ERR_INVALID_ARG;
    if (cfg->rows_capacity > 0 && (!Xp || !Gp || !H || !Yp)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({Xp, W1, b1, W2, b2, Gp, H, Yp})) return MOE_ERR_INVALID_ARG;
    if (cfg->rows_capacity == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const moe_config_t& c = *cfg;
    RowGemmArgs g1{};
    g1.kind = kGemmFfn1; g1.A = Xp; g1.B = W1; g1.bias = b1; g1.out0 = Gp; g1.out1 = H;
    g1.offsets = offsets; g1.E = c.E; g1.N = c.d_ff; g1.K = c.d; g1.rows_capacity = c.rows_capacity;
    g1.sBe = (long long)c.d_ff * c.d; g1.sBn = c.d; g1.sBk = 1;
    MOE_TRY(row_gemm(c, g1, s));
    RowGemmArgs g2{};
    g2.kind = kGemmFfn2; g2.A = H; g2.B = W2; g2.bias = b2; g2.out0 = Yp;
    g2.offsets = offsets; g2.E = c.E; g2.N = c.d; g2.K = c.d_ff; g2.rows_capacity = c.rows_capacity;
    g2.sBe = (long long)c.d * c.d_ff; g2.sBn = c.d_ff; g2.sBk = 1;
    MOE_TRY(row_gemm(c, g2, s));
    return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* Yp, const int32_t* slot_row,
                         const float* w, void* y, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (cfg->T > 0 && (!Yp || !slot_row || !w || !y)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({Yp, y})) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(*cfg, Yp, slot_row, w, y, (cudaStream_t)stream));
}

moe_status_t moe_backward(const moe_config_t* cfg, const void* dy, const void* x, const void* Wg,
                          const int32_t* idx, const float* w, const int32_t* offsets,
                          const int32_t* row_token, const int32_t* slot_row, const void* Xp,
                          const void* Gp, const void* H, const void* Yp, const void* W1,
                          const void* W2, const float* balance_loss, void* dx, float* dWg, void* dW1,
                          float* db1, void* dW2, float* db2, float* dbg, float* dw, float* loss,
                          void* ws, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!Wg || !offsets || !W1 || !W2 || !dWg || !dW1 || !db1 || !dW2 || !db2 || !ws)
        return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!dy || !x || !idx || !w || !slot_row || !dx)) return MOE_ERR_INVALID_ARG;
    if (cfg->rows_capacity > 0 && (!row_token || !Xp || !Gp || !H || !Yp)) return MOE_ERR_INVALID_ARG;
    if (!aligned16({dy, x, Wg, Xp, Gp, H, Yp, W1, W2, dx, dW1, dW2, ws})) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = *cfg;
    cudaStream_t s = (cudaStream_t)stream;
    BackwardScratch b;
    carve_backward(c, ws, &b);
    float* dwp = dw ? dw : b.dw;

    cudaStream_t side = side_stream();
    if (!side) return MOE_ERR_CUDA;
    // With a kernel trace open on this thread the main stream also waits for the side branch
    // before dH and before dX, so that no two kernels overlap and each traced duration is the
    // kernel's own, not a wait for SMs held by the other branch.
    const bool serial = t_trace_on;

    // The backward is a small DAG.
    //   main: combine backward -> dH -> dX -> un-permute (dx)
    //   side: dz (softmax Jacobian) + loss -> dWg, dbg -> dW2, db2 -> [after dH] dW1, db1
    // dz needs only the combine backward's dw, so where dz^T x runs on the tensor cores
    // (bf16, more than 32 experts, or dense routing) dz and the gate-weight gradient run
    // beside the expert GEMMs and only the un-permute follows dX. With 32 experts or fewer the
    // CUDA-core dz^T x kernels would take SMs from dH (measured 2% slower that way): the
    // router backward and dz^T x follow dX on the main stream, from dense dz rows. Otherwise
    // (no tensor cores, more than 32 experts) the assignments are sorted by expert after dX.
    // The branches fork and join through events, which also works under stream capture; they
    // write disjoint outputs, so results do not depend on the overlap.
    EventSet ev(serial);
    if (!ev.ok) return MOE_ERR_CUDA;
    float* dbg_out = c.has_gate_bias ? dbg : nullptr;
    const bool early_dz = dense_routing(c) || (c.dtype == MOE_BF16 && c.d % 64 == 0 && c.E > 32);
    float* dz_dense = dense_routing(c) ? b.dz : b.soft.dz;

    // combine backward: dYp, dw, loss partials (padding rows of dYp zeroed)
    MOE_TRY(launch_combine_bwd(c, dy, Yp, w, offsets, row_token, slot_row, b.dYp, dwp, b.lossblk, s));
    MOE_TRY(cudaEventRecord(ev.a, s));
    MOE_TRY(cudaStreamWaitEvent(side, ev.a, 0));
    if (early_dz) {
        MOE_TRY(launch_router_dz(c, w, dwp, idx, b.dz, dense_routing(c) ? nullptr : dz_dense, b.lossblk,
                                 balance_loss, loss, side));
        MOE_TRY(cudaEventRecord(ev.d, side));
        MOE_TRY(launch_dense_dwg(c, dz_dense, x, dWg, dbg_out, false, b.soft, side));
    }
    // the weight gradients' K loops stop at each bucket's last row with an assignment
    if (use_tc(c)) MOE_TRY(launch_bucket_used(c, offsets, row_token, b.used, side));
    WgradArgs w2{b.dYp, H, dW2, offsets, c.E, c.d, c.d_ff};
    if (use_tc(c)) w2.rows_used = b.used;
    MOE_TRY(wgrad(c, w2, side));
    MOE_TRY(launch_colsum(c, b.dYp, c.d, offsets, b.colsum_d, side));
    MOE_TRY(launch_bias_reduce(c, b.colsum_d, c.d, offsets, db2, side));
    if (serial) {
        MOE_TRY(cudaEventRecord(ev.e, side));
        MOE_TRY(cudaStreamWaitEvent(s, ev.e, 0));
    }
    // experts backward on the main stream
    RowGemmArgs gh{};
    gh.kind = kGemmDH; gh.A = b.dYp; gh.B = W2; gh.aux = Gp; gh.out0 = b.dA;
    gh.colsum = use_tc(c) ? b.colsum_f : nullptr;  // the tensor-core epilogue sums dA columns
    gh.offsets = offsets; gh.E = c.E; gh.N = c.d_ff; gh.K = c.d; gh.rows_capacity = c.rows_capacity;
    gh.sBe = (long long)c.d * c.d_ff; gh.sBn = 1; gh.sBk = c.d_ff;
    MOE_TRY(row_gemm(c, gh, s));
    if (!use_tc(c)) MOE_TRY(launch_colsum(c, b.dA, c.d_ff, offsets, b.colsum_f, s));
    MOE_TRY(cudaEventRecord(ev.b, s));
    MOE_TRY(cudaStreamWaitEvent(side, ev.b, 0));
    WgradArgs w1{b.dA, Xp, dW1, offsets, c.E, c.d_ff, c.d};
    if (use_tc(c)) w1.rows_used = b.used;
    MOE_TRY(wgrad(c, w1, side));
    MOE_TRY(launch_bias_reduce(c, b.colsum_f, c.d_ff, offsets, db1, side));
    if (serial) {
        MOE_TRY(cudaEventRecord(ev.f, side));
        MOE_TRY(cudaStreamWaitEvent(s, ev.f, 0));
    }
    RowGemmArgs gx{};
    gx.kind = kGemmDX; gx.A = b.dA; gx.B = W1; gx.out0 = b.dXp;
    gx.offsets = offsets; gx.E = c.E; gx.N = c.d; gx.K = c.d_ff; gx.rows_capacity = c.rows_capacity;
    gx.sBe = (long long)c.d_ff * c.d; gx.sBn = 1; gx.sBk = c.d;
    MOE_TRY(row_gemm(c, gx, s));
    if (early_dz) {
        // un-permute: dx = sum over kept slots of dXp rows + dz Wg, with dz from the side branch
        MOE_TRY(cudaStreamWaitEvent(s, ev.d, 0));
        MOE_TRY(launch_router_bwd(c, w, dwp, idx, slot_row, Wg, b.dXp, b.dz, dx, nullptr, nullptr, nullptr,
                                  nullptr, true, s));
    } else if (c.E <= 32) {
        MOE_TRY(launch_router_bwd(c, w, dwp, idx, slot_row, Wg, b.dXp, b.dz, dx, dz_dense, b.lossblk,
                                  balance_loss, loss, false, s));
        MOE_TRY(launch_dense_dwg(c, dz_dense, x, dWg, dbg_out, false, b.soft, s));
    } else {
        MOE_TRY(launch_sort(c, idx, b.sort, nullptr, nullptr, nullptr, nullptr, nullptr, s));
        MOE_TRY(launch_router_bwd(c, w, dwp, idx, slot_row, Wg, b.dXp, b.dz, dx, nullptr, b.lossblk,
                                  balance_loss, loss, false, s));
        MOE_TRY(launch_dwg(c, x, b.dz, b.sort, b.dwg_part, dWg, dbg_out, s));
    }
    // join
    MOE_TRY(cudaEventRecord(ev.c, side));
    MOE_TRY(cudaStreamWaitEvent(s, ev.c, 0));
    return MOE_OK;
}

moe_status_t moe_coselect(const moe_config_t* cfg, const int32_t* idx, int32_t* H, moe_stream_t stream) {
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!H || (cfg->T > 0 && !idx)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_coselect(*cfg, idx, H, (cudaStream_t)stream));
}

moe_status_t moe_get_error(moe_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    int* p = device_error_word();
    if (!p) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v != kErrNone) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (v == kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (v == kErrBounds) return MOE_ERR_DEVICE_BOUNDS;
    return MOE_OK;
}

const char* moe_status_str(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_BOUNDS: return "index out of range on the device";
    }
    return "unknown status";
}

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_version(void) { return "moe-gb300 0.1 sm_103a"; }

}  // extern "C"
