// Combine (forward), combine backward, router backward + un-permute, gate-weight gradient,
// bias gradients and the reported loss.
//
// "Native MoE training system PithTrain", section 4.1: output[mask] += expert_output *
// routing_weight (weighted accumulate back to token order); section 4.2: loss.backward().
// "Expert Parallelism: Scaling Mixture-of-Experts Models", section 2.2: the weights are
// softmax(z / temperature) over the selected logits, whose Jacobian carries the gradient
// to the gate. "PyTorch distributed MoE training", section 4.3: aux_loss_weight * balance.
//
// All reductions run in a fixed order (no floating-point atomics), so results are
// bit-reproducible from run to run.
#include "internal.cuh"

namespace moe {

namespace {

// y[t] = sum over kept slots of w[t,j] * Yp[slot_row[t,j]]; one warp per token. Slots are
// taken in groups of G (one group unless k > G, i.e. dense routing), in slot order; G is the
// smallest of 1, 2, 4, 8 that holds k, so that the registers (and occupancy) follow k.
template <typename T, int G>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ Yp, const int32_t* __restrict__ slot_row,
               const float* __restrict__ w, int Tn, int d, int k, T* __restrict__ y) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        int rows[G];
        float ws[G];
        // the first group stays in registers across the column loop
#pragma unroll
        for (int j = 0; j < G; ++j) {
            rows[j] = (j < k) ? slot_row[(size_t)t * k + j] : -1;
            ws[j] = (j < k) ? w[(size_t)t * k + j] : 0.f;
        }
        if ((d % V) == 0) {
            // two column groups per pass, every row load of a slot group issued before any arithmetic
#pragma unroll 1
            for (int c = lane * V; c < d; c += 64 * V) {
                const int c2 = c + 32 * V;
                const bool two = c2 < d;
                float acc[2][V];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[h][i] = 0.f;
#pragma unroll 1
                for (int j0 = 0; j0 < k; j0 += G) {
                    int rg[G];
                    float wg[G];
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        if (j0 == 0) { rg[j] = rows[j]; wg[j] = ws[j]; }
                        else {
                            rg[j] = (j0 + j < k) ? slot_row[(size_t)t * k + j0 + j] : -1;
                            wg[j] = (j0 + j < k) ? w[(size_t)t * k + j0 + j] : 0.f;
                        }
                    }
                    uint4 raw[2][G];
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        if (rg[j] >= 0) {
                            raw[0][j] = __ldg(reinterpret_cast<const uint4*>(Yp + (size_t)rg[j] * d + c));
                            if (two) raw[1][j] = __ldg(reinterpret_cast<const uint4*>(Yp + (size_t)rg[j] * d + c2));
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !two) break;
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            if (rg[j] >= 0) {
                                float v[V];
                                unpack16<T>(raw[h][j], v);
#pragma unroll
                                for (int i = 0; i < V; ++i) acc[h][i] = fmaf(wg[j], v[i], acc[h][i]);
                            }
                        }
                    }
                }
                store16(y + (size_t)t * d + c, acc[0]);
                if (two) store16(y + (size_t)t * d + c2, acc[1]);
            }
        } else {
            for (int c = lane; c < d; c += 32) {
                float acc = 0.f;
                for (int j = 0; j < k; ++j) {
                    const int r = j < G ? rows[j] : slot_row[(size_t)t * k + j];
                    const float wj = j < G ? ws[j] : w[(size_t)t * k + j];
                    if (r >= 0) acc = fmaf(wj, ld_f(Yp + (size_t)r * d + c), acc);
                }
                st_f(y + (size_t)t * d + c, acc);
            }
        }
    }
}

// Zero the padding rows (row_token = -1) of a bucket buffer M [rows, d], rows < offsets[E]:
// each warp takes 32 rows at a time, finds the padding ones with a ballot and clears them
// together (coalesced 16-byte stores).
template <typename T>
__device__ __forceinline__ void zero_padding_rows(const int32_t* __restrict__ offsets, int E,
                                                  const int32_t* __restrict__ row_token, int d, int rows_cap,
                                                  T* __restrict__ M, int gw, int nwarps, int lane) {
    constexpr int V = Vec16<T>::N;
    const int nrows = min(offsets[E], rows_cap);
    for (int r0 = gw * 32; r0 < nrows; r0 += nwarps * 32) {
        const int r = r0 + lane;
        unsigned pad = __ballot_sync(0xffffffffu, r < nrows && row_token[r] < 0);
        while (pad) {
            const int b = __ffs(pad) - 1;
            pad &= pad - 1;
            T* out = M + (size_t)(r0 + b) * d;
            if ((d % V) == 0) {
                float z[V];
#pragma unroll
                for (int i = 0; i < V; ++i) z[i] = 0.f;
                for (int c = lane * V; c < d; c += 32 * V) store16(out + c, z);
            } else {
                for (int c = lane; c < d; c += 32) st_f(out + c, 0.f);
            }
        }
    }
}

// Combine backward, one warp per token, slots in groups of G (as in the combine):
//   kept slot j (row r):  dYp[r] = w[t,j] dy[t],  dw[t,j] = <dy[t], Yp[r]>
//   dropped slot j:       dw[t,j] = 0
// then the padding rows of dYp are zeroed. lossblk[block] = the block's sum of w * dw over
// kept slots (warps in order; a warp's tokens in order), so sum(lossblk) = sum_t <y[t], dy[t]>.
template <typename T, int G>
__global__ void __launch_bounds__(256, G >= 8 ? 2 : 1)
combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ Yp, const float* __restrict__ w,
                   const int32_t* __restrict__ offsets, int E, const int32_t* __restrict__ row_token,
                   const int32_t* __restrict__ slot_row, int Tn, int d, int k, int rows_cap,
                   T* __restrict__ dYp, float* __restrict__ dw, float* __restrict__ lossblk) {
    pdl_wait();
    __shared__ float s_warp[8];
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    float wloss = 0.f;
    for (int t = gw; t < Tn; t += nwarps) {
        for (int j0 = 0; j0 < k; j0 += G) {
            int rows[G];
            float ws[G], dot[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const bool in = j0 + j < k;
                rows[j] = in ? slot_row[(size_t)t * k + j0 + j] : -1;
                ws[j] = in ? w[(size_t)t * k + j0 + j] : 0.f;
                dot[j] = 0.f;
            }
            if ((d % V) == 0) {
                for (int c = lane * V; c < d; c += 32 * V) {
                    // the dy vector and every kept slot's Yp vector in flight before any arithmetic
                    const uint4 graw = __ldg(reinterpret_cast<const uint4*>(dy + (size_t)t * d + c));
                    uint4 yraw[G];
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (rows[j] >= 0) yraw[j] = __ldg(reinterpret_cast<const uint4*>(Yp + (size_t)rows[j] * d + c));
                    float g[V];
                    unpack16<T>(graw, g);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        if (rows[j] < 0) continue;
                        float yv[V], o[V];
                        unpack16<T>(yraw[j], yv);
#pragma unroll
                        for (int i = 0; i < V; ++i) { dot[j] = fmaf(g[i], yv[i], dot[j]); o[i] = ws[j] * g[i]; }
                        store16(dYp + (size_t)rows[j] * d + c, o);
                    }
                }
            } else {
                for (int c = lane; c < d; c += 32) {
                    const float g = ld_f(dy + (size_t)t * d + c);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        if (rows[j] < 0) continue;
                        dot[j] = fmaf(g, ld_f(Yp + (size_t)rows[j] * d + c), dot[j]);
                        st_f(dYp + (size_t)rows[j] * d + c, ws[j] * g);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float v = warp_sum(dot[j]);
                if (j0 + j < k) {
                    if (lane == 0) dw[(size_t)t * k + j0 + j] = rows[j] >= 0 ? v : 0.f;
                    if (rows[j] >= 0) wloss = fmaf(ws[j], v, wloss);
                }
            }
        }
    }
    zero_padding_rows(offsets, E, row_token, d, rows_cap, dYp, gw, nwarps, lane);
    if (lane == 0) s_warp[threadIdx.x >> 5] = wloss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b += s_warp[i];
        lossblk[blockIdx.x] = b;
    }
}

// loss = sum of the combine-backward block partials (fixed order) + aux * balance_loss, by
// the 256 threads of one block (every thread of the block must call it).
struct LossArgs {
    const float* lossblk;
    int nblk;
    const float* balance;
    float aux;
    float* loss;     // null: no loss
};
__device__ __forceinline__ void block_loss(const LossArgs& la) {
    __shared__ float red[8];
    float acc = 0.f;
    for (int i = threadIdx.x; i < la.nblk; i += blockDim.x) acc += la.lossblk[i];
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < 8; ++i) t += red[i];
        *la.loss = t + (la.balance ? la.aux * *la.balance : 0.f);
    }
}

// The softmax Jacobian of the routing weights alone, one warp per token (any k):
//   s = sum_j w_j dw_j,  dz_j = w_j (dw_j - s) / temperature  -> dz [T, k]
// and, when dz_dense is set (k <= MOE_MAX_K), dz as dense [T, E] rows (0 where unselected).
// Block 0 then writes the reported loss. It needs only combine-backward outputs, so it runs
// beside the expert GEMMs; the un-permute (dx) follows the dX GEMM.
__global__ void __launch_bounds__(256)
router_dz_kernel(const float* __restrict__ w, const float* __restrict__ dw, const int32_t* __restrict__ idx,
                 int Tn, int k, int E, float inv_temp, float* __restrict__ dz, float* __restrict__ dz_dense,
                 LossArgs la) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        const size_t base = (size_t)t * k;
        float sp = 0.f;
        for (int j = lane; j < k; j += 32) sp = fmaf(w[base + j], dw[base + j], sp);
        const float s = warp_sum(sp);
        for (int j = lane; j < k; j += 32) dz[base + j] = w[base + j] * (dw[base + j] - s) * inv_temp;
        if (dz_dense) {
            for (int e = lane; e < E; e += 32) {
                float v = 0.f;
                for (int j = 0; j < k; ++j)
                    if (idx[base + j] == e) v = w[base + j] * (dw[base + j] - s) * inv_temp;
                dz_dense[(size_t)t * E + e] = v;
            }
        }
    }
    if (blockIdx.x == 0 && la.loss) block_loss(la);   // whole block 0, after its tokens
}

// Router backward + un-permute, one warp per token (KC >= k slots held in registers):
//   s = sum_j w_j dw_j,  dz_j = w_j (dw_j - s) / temperature          (softmax Jacobian)
//   dx[t] = sum_{kept j} dXp[slot_row[t,j]] + sum_j dz_j Wg[idx[t,j]]
template <typename T, int KC>
__global__ void __launch_bounds__(256, KC >= 8 ? 2 : 1)
router_bwd_kernel(const float* __restrict__ w, const float* __restrict__ dw,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ slot_row,
                  const T* __restrict__ Wg, const T* __restrict__ dXp, int Tn, int d, int k,
                  int E, float inv_temp, float* __restrict__ dz, T* __restrict__ dx,
                  float* __restrict__ dz_dense, LossArgs la, bool dz_in) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        float wj[KC], dzj[KC];
        int rows[KC], ex[KC];
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            wj[j] = (j < k) ? w[(size_t)t * k + j] : 0.f;
            dzj[j] = (j < k) ? dw[(size_t)t * k + j] : 0.f;
            rows[j] = (j < k) ? slot_row[(size_t)t * k + j] : -1;
            ex[j] = (j < k) ? idx[(size_t)t * k + j] : 0;
            ex[j] = min(max(ex[j], 0), E - 1);
            s = fmaf(wj[j], dzj[j], s);
        }
#pragma unroll
        for (int j = 0; j < KC; ++j) dzj[j] = dz_in ? ((j < k) ? dz[(size_t)t * k + j] : 0.f)
                                                   : wj[j] * (dzj[j] - s) * inv_temp;
        if (lane < k && !dz_in) {
            float mine = 0.f;
#pragma unroll
            for (int j = 0; j < KC; ++j)
                if (j == lane) mine = dzj[j];
            dz[(size_t)t * k + lane] = mine;
        }
        if (dz_dense && lane < E) {
            // E <= 32: lane e writes expert e's entry of the dense [T, E] row (0 if unselected)
            float v = 0.f;
#pragma unroll
            for (int j = 0; j < KC; ++j)
                if (j < k && ex[j] == lane) v = dzj[j];
            dz_dense[(size_t)t * E + lane] = v;
        }
        if ((d % V) == 0) {
            for (int c = lane * V; c < d; c += 32 * V) {
                // every slot's dXp and Wg vectors in flight before any arithmetic, then the same
                // order of additions as one slot at a time
                uint4 xraw[KC], graw[KC];
#pragma unroll
                for (int j = 0; j < KC; ++j) {
                    if (j < k) {
                        if (rows[j] >= 0) xraw[j] = __ldg(reinterpret_cast<const uint4*>(dXp + (size_t)rows[j] * d + c));
                        graw[j] = __ldg(reinterpret_cast<const uint4*>(Wg + (size_t)ex[j] * d + c));
                    }
                }
                float acc[V];
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
                for (int j = 0; j < KC; ++j) {
                    if (j < k) {
                        float v[V];
                        if (rows[j] >= 0) {
                            unpack16<T>(xraw[j], v);
#pragma unroll
                            for (int i = 0; i < V; ++i) acc[i] += v[i];
                        }
                        unpack16<T>(graw[j], v);
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[i] = fmaf(dzj[j], v[i], acc[i]);
                    }
                }
                store16(dx + (size_t)t * d + c, acc);
            }
        } else {
            for (int c = lane; c < d; c += 32) {
                float acc = 0.f;
                for (int j = 0; j < k; ++j) {
                    if (rows[j] >= 0) acc += ld_f(dXp + (size_t)rows[j] * d + c);
                    acc = fmaf(dzj[j], ld_f(Wg + (size_t)ex[j] * d + c), acc);
                }
                st_f(dx + (size_t)t * d + c, acc);
            }
        }
    }
    if (blockIdx.x == 0 && la.loss) block_loss(la);   // whole block 0, after its tokens
}

// Router backward + un-permute for k > MOE_MAX_K (dense routing, k = E): one warp per token,
// the token's k slots staged in shared memory (s and the dz values lane-parallel), then per
// column group the same order as router_bwd_kernel: for each slot j, add dXp[row_j], then
// dz_j Wg[e_j]. Four slots' loads are issued before their arithmetic.
template <typename T>
__global__ void __launch_bounds__(256)
router_bwd_wide_kernel(const float* __restrict__ w, const float* __restrict__ dw,
                       const int32_t* __restrict__ idx, const int32_t* __restrict__ slot_row,
                       const T* __restrict__ Wg, const T* __restrict__ dXp, int Tn, int d, int k,
                       int E, float inv_temp, float* __restrict__ dz, T* __restrict__ dx, LossArgs la,
                       bool dz_in) {
    pdl_wait();
    __shared__ float s_dz[8][MOE_MAX_EXPERTS];
    __shared__ int s_row[8][MOE_MAX_EXPERTS];
    __shared__ int s_ex[8][MOE_MAX_EXPERTS];
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    constexpr int V = Vec16<T>::N;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
        const size_t base = (size_t)t * k;
        float s = 0.f;
        for (int j = lane; j < k; j += 32) s = fmaf(w[base + j], dw[base + j], s);
        s = warp_sum(s);
        for (int j = lane; j < k; j += 32) {
            const float v = dz_in ? dz[base + j] : w[base + j] * (dw[base + j] - s) * inv_temp;
            s_dz[wid][j] = v;
            if (!dz_in) dz[base + j] = v;
            s_row[wid][j] = slot_row[base + j];
            s_ex[wid][j] = min(max(idx[base + j], 0), E - 1);
        }
        __syncwarp();
        const float* zj = s_dz[wid];
        const int* rj = s_row[wid];
        const int* ej = s_ex[wid];
        if ((d % V) == 0) {
            for (int c = lane * V; c < d; c += 32 * V) {
                float acc[V];
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = 0.f;
                int j = 0;
                for (; j + 4 <= k; j += 4) {
                    float xr[4][V], wr[4][V];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (rj[j + u] >= 0) load16(dXp + (size_t)rj[j + u] * d + c, xr[u]);
                        else {
#pragma unroll
                            for (int i = 0; i < V; ++i) xr[u][i] = 0.f;
                        }
                        load16(Wg + (size_t)ej[j + u] * d + c, wr[u]);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            if (rj[j + u] >= 0) acc[i] += xr[u][i];
                            acc[i] = fmaf(zj[j + u], wr[u][i], acc[i]);
                        }
                    }
                }
                for (; j < k; ++j) {
                    float v[V];
                    if (rj[j] >= 0) {
                        load16(dXp + (size_t)rj[j] * d + c, v);
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[i] += v[i];
                    }
                    load16(Wg + (size_t)ej[j] * d + c, v);
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[i] = fmaf(zj[j], v[i], acc[i]);
                }
                store16(dx + (size_t)t * d + c, acc);
            }
        } else {
            for (int c = lane; c < d; c += 32) {
                float acc = 0.f;
                for (int j = 0; j < k; ++j) {
                    if (rj[j] >= 0) acc += ld_f(dXp + (size_t)rj[j] * d + c);
                    acc = fmaf(zj[j], ld_f(Wg + (size_t)ej[j] * d + c), acc);
                }
                st_f(dx + (size_t)t * d + c, acc);
            }
        }
        __syncwarp();
    }
    if (blockIdx.x == 0 && la.loss) block_loss(la);   // whole block 0, after its tokens
}

// dWg partials: block (e, chunk) sums dz[a] * x[token(a)] over a contiguous piece of expert
// e's assignment segment, in segment order. The piece's token ids and dz values are staged in
// shared memory; each thread owns V consecutive columns and keeps 8 row loads in flight.
template <typename T>
__global__ void __launch_bounds__(256)
dwg_partial_kernel(const T* __restrict__ x, const float* __restrict__ dz,
                   const int32_t* __restrict__ assign_off, const int32_t* __restrict__ assign_tok,
                   int d, int k, int nchunk, float* __restrict__ part) {
    pdl_wait();
    constexpr int V = Vec16<T>::N;
    constexpr int PIECE = 256;
    __shared__ int s_tok[PIECE];
    __shared__ float s_dz[PIECE];
    const int e = blockIdx.y, chunk = blockIdx.x;
    const int seg0 = assign_off[e], seg1 = assign_off[e + 1];
    const int per = (seg1 - seg0 + nchunk - 1) / nchunk;
    const int a0 = seg0 + chunk * per, a1 = min(seg1, a0 + per);
    float* out = part + ((size_t)e * nchunk + chunk) * d;
    const bool vec = (d % V) == 0;
    const int step = vec ? V : 1;
    // every thread runs the same number of passes: the barriers below are block-wide
    const int passes = (d + (int)blockDim.x * step - 1) / ((int)blockDim.x * step);
    for (int pass = 0; pass < passes; ++pass) {
        const int cg = (pass * (int)blockDim.x + (int)threadIdx.x) * step;
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        const bool active = cg < d;
        for (int p0 = a0; p0 < a1; p0 += PIECE) {
            const int n = min(PIECE, a1 - p0);
            __syncthreads();
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int at = assign_tok[p0 + i];
                s_tok[i] = at / k;
                s_dz[i] = dz[at];
            }
            __syncthreads();
            if (!active) continue;
            if (vec) {
                int i = 0;
                for (; i + 8 <= n; i += 8) {
                    float v[8][V];
#pragma unroll
                    for (int u = 0; u < 8; ++u) load16(x + (size_t)s_tok[i + u] * d + cg, v[u]);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
#pragma unroll
                        for (int q = 0; q < V; ++q) acc[q] = fmaf(s_dz[i + u], v[u][q], acc[q]);
                }
                for (; i < n; ++i) {
                    float v[V];
                    load16(x + (size_t)s_tok[i] * d + cg, v);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[q] = fmaf(s_dz[i], v[q], acc[q]);
                }
            } else {
                for (int i = 0; i < n; ++i) acc[0] = fmaf(s_dz[i], ld_f(x + (size_t)s_tok[i] * d + cg), acc[0]);
            }
        }
        if (active) {
            if (vec) {
#pragma unroll
                for (int q = 0; q < V; ++q) out[cg + q] = acc[q];
            } else {
                out[cg] = acc[0];
            }
        }
    }
}

// dWg[e, c] = sum over chunks of the partials (fixed order); dbg[e] = sum of dz over e's
// assignments (one block per expert, fixed reduction tree).
__global__ void __launch_bounds__(256)
dwg_reduce_kernel(const float* __restrict__ part, int d, int nchunk, float* __restrict__ dWg) {
    pdl_wait();
    const int e = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= d) return;
    float acc = 0.f;
    for (int ch = 0; ch < nchunk; ++ch) acc += part[((size_t)e * nchunk + ch) * d + c];
    dWg[(size_t)e * d + c] = acc;
}

__global__ void __launch_bounds__(256)
dbg_kernel(const float* __restrict__ dz, const int32_t* __restrict__ assign_off,
           const int32_t* __restrict__ assign_tok, float* __restrict__ dbg) {
    pdl_wait();
    __shared__ float red[256];
    const int e = blockIdx.x;
    float acc = 0.f;
    for (int a = assign_off[e] + threadIdx.x; a < assign_off[e + 1]; a += blockDim.x)
        acc += dz[assign_tok[a]];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) dbg[e] = red[0];
}

// Column sums of one 32-row quarter of a 128-row tile (tiles never straddle buckets;
// padding rows are zero): part[tile * 4 + quarter, c] = sum of M[r, c] over the quarter's rows.
template <typename T>
__global__ void __launch_bounds__(256)
colsum_quarter_kernel(const T* __restrict__ M, int width, const int32_t* __restrict__ offsets, int E,
                      float* __restrict__ part) {
    pdl_wait();
    constexpr int V = Vec16<T>::N;
    constexpr int QROWS = MOE_ROW_ALIGN / kColsumParts;
    const int pq = blockIdx.x;  // tile * 4 + quarter (x: up to 2^31 - 1 quarters)
    const int r0 = pq * QROWS;
    if (r0 >= offsets[E]) return;
    if (width % V == 0) {
        const int c = (blockIdx.y * blockDim.x + threadIdx.x) * V;
        if (c >= width) return;
        float acc[V];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll 8
        for (int r = 0; r < QROWS; ++r) {
            float v[V];
            load16(M + (size_t)(r0 + r) * width + c, v);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] += v[q];
        }
#pragma unroll
        for (int q = 0; q < V; ++q) part[(size_t)pq * width + c + q] = acc[q];
    } else {
        const int cend = min(width, (int)((blockIdx.y + 1) * blockDim.x * V));
        for (int c = blockIdx.y * blockDim.x * V + threadIdx.x; c < cend; c += blockDim.x) {
            float acc = 0.f;
            for (int r = 0; r < QROWS; ++r) acc += ld_f(M + (size_t)(r0 + r) * width + c);
            part[(size_t)pq * width + c] = acc;
        }
    }
}

// db[e, c] = sum over the quarters of bucket e's tiles of part[., c], in order.
__global__ void __launch_bounds__(256)
bias_reduce_kernel(const float* __restrict__ part, int width, const int32_t* __restrict__ offsets,
                   float* __restrict__ db) {
    pdl_wait();
    const int e = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= width) return;
    const int q0 = offsets[e] / MOE_ROW_ALIGN * kColsumParts, q1 = offsets[e + 1] / MOE_ROW_ALIGN * kColsumParts;
    float acc = 0.f;
    for (int q = q0; q < q1; ++q) acc += part[(size_t)q * width + c];
    db[(size_t)e * width + c] = acc;
}

// loss = sum of the combine-backward block partials (fixed order) + aux * balance_loss.
__global__ void __launch_bounds__(256)
loss_kernel(const float* __restrict__ lossblk, int nblk, const float* __restrict__ balance, float aux,
            float* __restrict__ loss) {
    pdl_wait();
    __shared__ float red[8];
    float acc = 0.f;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) acc += lossblk[i];
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < 8; ++i) t += red[i];
        *loss = t + (balance ? aux * *balance : 0.f);
    }
}

int warp_grid(long long items, int warps_per_block = 8) {
    long long b = (items + warps_per_block - 1) / warps_per_block;
    return (int)std::max(1LL, std::min(b, (long long)num_sms() * 16));
}

}  // namespace

template <typename T, int G>
static cudaError_t combine_g(const moe_config_t& c, const void* Yp, const int32_t* slot_row, const float* w,
                             void* y, cudaStream_t s) {
    const int grid = warp_grid(c.T);
    return launch_pdl(combine_kernel<T, G>, grid, 256, 0, s, (const T*)Yp, slot_row, w, c.T, c.d, c.k, (T*)y);
}
template <typename T>
static cudaError_t combine_t(const moe_config_t& c, const void* Yp, const int32_t* slot_row, const float* w,
                             void* y, cudaStream_t s) {
    if (c.k <= 1) return combine_g<T, 1>(c, Yp, slot_row, w, y, s);
    if (c.k <= 2) return combine_g<T, 2>(c, Yp, slot_row, w, y, s);
    if (c.k <= 4) return combine_g<T, 4>(c, Yp, slot_row, w, y, s);
    return combine_g<T, 8>(c, Yp, slot_row, w, y, s);
}

cudaError_t launch_combine(const moe_config_t& c, const void* Yp, const int32_t* slot_row,
                           const float* w, void* y, cudaStream_t s) {
    if (c.T == 0) return cudaSuccess;
    cudaError_t e = c.dtype == MOE_BF16 ? combine_t<__nv_bfloat16>(c, Yp, slot_row, w, y, s)
                                        : combine_t<float>(c, Yp, slot_row, w, y, s);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int combine_bwd_blocks(const moe_config_t& c) { return warp_grid(std::max(c.T, 1)); }

template <typename T, int G>
static cudaError_t combine_bwd_g(const moe_config_t& c, const void* dy, const void* Yp, const float* w,
                                 const int32_t* offsets, const int32_t* row_token, const int32_t* slot_row,
                                 void* dYp, float* dw, float* lossblk, cudaStream_t s) {
    return launch_pdl(combine_bwd_kernel<T, G>, combine_bwd_blocks(c), 256, 0, s, (const T*)dy, (const T*)Yp, w,
                      offsets, c.E, row_token, slot_row, c.T, c.d, c.k, c.rows_capacity, (T*)dYp, dw, lossblk);
}
template <typename T>
static cudaError_t combine_bwd_t(const moe_config_t& c, const void* dy, const void* Yp, const float* w,
                                 const int32_t* offsets, const int32_t* row_token, const int32_t* slot_row,
                                 void* dYp, float* dw, float* lossblk, cudaStream_t s) {
    if (c.k <= 1) return combine_bwd_g<T, 1>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s);
    if (c.k <= 2) return combine_bwd_g<T, 2>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s);
    if (c.k <= 4) return combine_bwd_g<T, 4>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s);
    return combine_bwd_g<T, 8>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s);
}

cudaError_t launch_combine_bwd(const moe_config_t& c, const void* dy, const void* Yp,
                               const float* w, const int32_t* offsets, const int32_t* row_token,
                               const int32_t* slot_row, void* dYp, float* dw, float* lossblk,
                               cudaStream_t s) {
    cudaError_t e = c.dtype == MOE_BF16
                        ? combine_bwd_t<__nv_bfloat16>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s)
                        : combine_bwd_t<float>(c, dy, Yp, w, offsets, row_token, slot_row, dYp, dw, lossblk, s);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T, int KC>
static void router_bwd_kc(const moe_config_t& c, int grid, float inv_temp, const float* w, const float* dw,
                          const int32_t* idx, const int32_t* slot_row, const void* Wg, const void* dXp, float* dz,
                          void* dx, float* dz_dense, const LossArgs& la, bool dz_in, cudaStream_t s) {
    launch_pdl(router_bwd_kernel<T, KC>, grid, 256, 0, s, w, dw, idx, slot_row, (const T*)Wg, (const T*)dXp, c.T, c.d,
               c.k, c.E, inv_temp, dz, (T*)dx, dz_dense, la, dz_in);
}
template <typename T>
static void router_bwd_narrow(const moe_config_t& c, int grid, float inv_temp, const float* w, const float* dw,
                              const int32_t* idx, const int32_t* slot_row, const void* Wg, const void* dXp, float* dz,
                              void* dx, float* dz_dense, const LossArgs& la, bool dz_in, cudaStream_t s) {
    if (c.k <= 1) router_bwd_kc<T, 1>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la, dz_in, s);
    else if (c.k <= 2) router_bwd_kc<T, 2>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la, dz_in, s);
    else if (c.k <= 4) router_bwd_kc<T, 4>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la, dz_in, s);
    else router_bwd_kc<T, 8>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la, dz_in, s);
}

cudaError_t launch_router_bwd(const moe_config_t& c, const float* w, const float* dw,
                              const int32_t* idx, const int32_t* slot_row, const void* Wg,
                              const void* dXp, float* dz, void* dx, float* dz_dense,
                              const float* lossblk, const float* balance_loss, float* loss, bool dz_in,
                              cudaStream_t s) {
    LossArgs la{lossblk, combine_bwd_blocks(c), balance_loss, c.aux_loss_weight, loss};
    if (c.T == 0) {
        if (loss) return launch_loss(c, lossblk, balance_loss, loss, s);
        return cudaSuccess;
    }
    const int grid = warp_grid(c.T);
    const float inv_temp = 1.0f / c.temperature;
    if (c.k > MOE_MAX_K) {
        if (c.dtype == MOE_BF16)
            launch_pdl(router_bwd_wide_kernel<__nv_bfloat16>, grid, 256, 0, s, w, dw, idx, slot_row,
                       (const __nv_bfloat16*)Wg, (const __nv_bfloat16*)dXp, c.T, c.d, c.k, c.E, inv_temp, dz,
                       (__nv_bfloat16*)dx, la, dz_in);
        else
            launch_pdl(router_bwd_wide_kernel<float>, grid, 256, 0, s, w, dw, idx, slot_row, (const float*)Wg,
                       (const float*)dXp, c.T, c.d, c.k, c.E, inv_temp, dz, (float*)dx, la, dz_in);
    } else if (c.dtype == MOE_BF16) {
        router_bwd_narrow<__nv_bfloat16>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la,
                                         dz_in, s);
    } else {
        router_bwd_narrow<float>(c, grid, inv_temp, w, dw, idx, slot_row, Wg, dXp, dz, dx, dz_dense, la, dz_in, s);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_router_dz(const moe_config_t& c, const float* w, const float* dw, const int32_t* idx,
                             float* dz, float* dz_dense, const float* lossblk, const float* balance_loss,
                             float* loss, cudaStream_t s) {
    if (c.T == 0) {
        if (loss) return launch_loss(c, lossblk, balance_loss, loss, s);
        return cudaSuccess;
    }
    LossArgs la{lossblk, combine_bwd_blocks(c), balance_loss, c.aux_loss_weight, loss};
    launch_pdl(router_dz_kernel, warp_grid(c.T), 256, 0, s, w, dw, idx, c.T, c.k, c.E, 1.0f / c.temperature, dz,
               dz_dense, la);
    count_launch();
    return cudaGetLastError();
}

int dwg_chunks(const moe_config_t& c) {
    // about four blocks per SM in total, each on a contiguous piece of one expert's segment
    int n = ceil_div(4LL * num_sms(), c.E);
    return std::max(1, std::min(n, 64));
}

cudaError_t launch_dwg(const moe_config_t& c, const void* x, const float* dz,
                       const SortScratch& srt, float* part, float* dWg, float* dbg, cudaStream_t s) {
    const int nchunk = dwg_chunks(c);
    dim3 g1(nchunk, c.E);
    const int V = c.dtype == MOE_BF16 ? 8 : 4;
    const int threads = std::max(32, std::min(256, (ceil_div(c.d, V) + 31) / 32 * 32));
    if (c.dtype == MOE_BF16)
        launch_pdl(dwg_partial_kernel<__nv_bfloat16>, g1, threads, 0, s, (const __nv_bfloat16*)x, dz, srt.assign_off,
                                                                 srt.assign_tok, c.d, c.k, nchunk, part);
    else
        launch_pdl(dwg_partial_kernel<float>, g1, threads, 0, s, (const float*)x, dz, srt.assign_off,
                                                         srt.assign_tok, c.d, c.k, nchunk, part);
    count_launch();
    dim3 g2(ceil_div(c.d, 256), c.E);
    launch_pdl(dwg_reduce_kernel, g2, 256, 0, s, part, c.d, nchunk, dWg);
    count_launch();
    if (dbg) {
        launch_pdl(dbg_kernel, c.E, 256, 0, s, dz, srt.assign_off, srt.assign_tok, dbg);
        count_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_colsum(const moe_config_t& c, const void* M, int width, const int32_t* offsets,
                          float* part, cudaStream_t s) {
    const int quarters = c.rows_capacity / MOE_ROW_ALIGN * kColsumParts;
    if (quarters == 0) return cudaSuccess;
    const int V = c.dtype == MOE_BF16 ? 8 : 4;
    const int threads = std::max(32, std::min(256, (ceil_div(width, V) + 31) / 32 * 32));
    dim3 g(quarters, ceil_div(width, threads * V));
    if (c.dtype == MOE_BF16)
        launch_pdl(colsum_quarter_kernel<__nv_bfloat16>, g, threads, 0, s, (const __nv_bfloat16*)M, width, offsets, c.E, part);
    else
        launch_pdl(colsum_quarter_kernel<float>, g, threads, 0, s, (const float*)M, width, offsets, c.E, part);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_bias_reduce(const moe_config_t& c, const float* part, int width,
                               const int32_t* offsets, float* db, cudaStream_t s) {
    dim3 g(ceil_div(width, 256), c.E);
    launch_pdl(bias_reduce_kernel, g, 256, 0, s, part, width, offsets, db);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_loss(const moe_config_t& c, const float* lossblk, const float* balance_loss,
                        float* loss, cudaStream_t s) {
    launch_pdl(loss_kernel, 1, 256, 0, s, lossblk, combine_bwd_blocks(c), balance_loss, c.aux_loss_weight, loss);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
