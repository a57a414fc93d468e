"""Plain CPU fp64 oracle of the MoE layer: token routing and expert compute, forward and backward.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline /
reference legs may import or call this module. The product path (the CUDA library and its
Python binding) never imports it and shares no code with it; the two meet only through
the seeded input generators in synth/.

Sources (pages cited by title and section):
* "Native MoE training system PithTrain" (PithTrain page), section 4.1: PithTrainMoELayer
  (gate Linear(dim, num_experts, bias=False); torch.topk(logits, k=2) then softmax over the
  selected values; experts Linear(dim, 4 dim) -> GELU -> Linear(4 dim, dim); routing-weighted
  accumulate back to token order); section 4.3 item 1 (capacity = capacity_factor *
  tokens_per_batch / num_experts, overflow tokens dropped).
* "PyTorch distributed MoE training" (PyTorch-MoE page), section 2.3 (DistributedMoELayer:
  softmax over all experts then argmax), section 3.2 (Expert: linear2(gelu(linear1(x))) with
  nn.Linear biases), section 3.3 (balance_loss: load by scatter_add of ones, then
  mean((load - mean(load))^2)), section 4.3 (aux_loss_weight = 0.01).
* "Expert Parallelism: Scaling Mixture-of-Experts Models" (Expert-Parallelism page),
  section 2.2 (g = softmax(gate(x) / temperature), y = sum_i g_i expert_i(x); hybrid: top-8
  pre-selection then soft weights over those 8), section 2.3 (load statistics averaged over a
  sliding window of the last 100 batches), section 4.2 idea 2 (tokens written straight into
  per-expert bucket offsets), section 5.5 (routing in FP32 precision).

Readings where the pages are silent or ambiguous:
* weights: top-k on logits, then softmax(z_sel / temperature) over the k selected (PithTrain
  4.1; temperature 1 for plain top-k). Indices equal those of softmax-then-top-k.
* ties in top-k go to the lower expert id; slot j holds the j-th largest logit.
* k = E is dense soft routing (the naive soft MoE): every expert on every token, slot j
  holds expert j, weights softmax(z / temperature) over all E.
* capacity C = ceil(capacity_factor * T * k / E) (tokens read as routed assignments),
  evaluated in IEEE double from the fp32 value of capacity_factor.
* drop priority: token order; assignment (t, j) -> e has rank = number of earlier tokens
  that picked e; kept iff rank < C. Dropped assignments add 0 to y; the surviving weights
  are not renormalised.
* balance loss counts are the router's pre-capacity choices (all T*k assignments); it has
  no gradient (integer counts).
* GELU is the exact erf form (nn.GELU default).
* the loss the layer reports is sum(y * dy) + aux_loss_weight * balance_loss; dy is the
  gradient seed.
* sliding window: the window holds the soft loads of the current batch and the W - 1 batches
  before it (all batches so far until W have been seen); the loss is the soft balance loss of
  their mean, and its gradient reaches only the current batch (earlier batches are stored
  statistics).

Every function below is pinned by tests/test_oracle_pins.py and tests/test_oracle_grad.py
against closed forms, hand-worked examples (tests/golden/), brute force on tiny inputs and
central finite differences; none is parity-unpinned.
"""
import math

import numpy as np
from scipy.special import erf

AUX_LOSS_WEIGHT = 0.01  # PyTorch-MoE page, section 4.3


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------- routing

def gate_logits(x, Wg, bg=None):
    """z = x Wg^T (+ bg): the gate linear (PithTrain page 4.1; PyTorch-MoE page 2.3), in fp64."""
    z = _f64(x) @ _f64(Wg).T
    if bg is not None:
        z = z + _f64(bg)[None, :]
    return z


def select_topk(z, k):
    """Indices of the k largest logits per token, largest first, ties to the lower expert id
    (torch.topk, PithTrain page 4.1). Returns (idx [T,k] int64, z_sel [T,k])."""
    z = _f64(z)
    order = np.argsort(-z, axis=1, kind="stable")  # stable: equal logits keep ascending id
    idx = order[:, :k].astype(np.int64)
    return idx, np.take_along_axis(z, idx, axis=1)


def select_all(z):
    """Dense soft routing, k = E (Expert-Parallelism page 2.2, the naive soft MoE that runs every
    expert on every token): nothing is selected, so slot j holds expert j and z_sel = z. No
    rounding can change the selection: the returned gap is +inf for every token.
    Returns (idx [T,E] int64, z_sel [T,E], gap [T])."""
    z = _f64(z)
    T, E = z.shape
    idx = np.broadcast_to(np.arange(E, dtype=np.int64), (T, E)).copy()
    return idx, z.copy(), np.full(T, np.inf)


def topk_gap(z, k):
    """Smallest difference between neighbours among the k+1 largest logits of each token.
    A token whose gap is tiny can flip its selection or slot order under rounding."""
    z = _f64(z)
    T, E = z.shape
    m = min(k + 1, E)
    if m < 2:
        return np.full(T, np.inf)
    s = -np.sort(-z, axis=1)[:, :m]
    return (s[:, :-1] - s[:, 1:]).min(axis=1)


def routing_weights(z_sel, temperature=1.0):
    """softmax(z_sel / temperature) over the k selected logits (PithTrain page 4.1 softmax over
    the top-k values; Expert-Parallelism page 2.2 temperature softmax over a top-8 set)."""
    s = _f64(z_sel) / float(temperature)
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=1, keepdims=True)


def expert_counts(idx, E):
    """load[e] = number of (token, slot) assignments to expert e (PyTorch-MoE page 3.3:
    load.scatter_add_(0, expert_indices, ones))."""
    return np.bincount(np.asarray(idx).reshape(-1), minlength=E).astype(np.int64)


def balance_loss(counts):
    """mean over experts of (load - mean(load))^2 (PyTorch-MoE page 3.3, balance_loss)."""
    load = np.asarray(counts, dtype=np.float64)
    return float(np.mean((load - load.mean()) ** 2))


# ----------------------------------------------------------------------------- routing noise

_PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
_PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)
_U64 = (1 << 64) - 1


def philox4x64_10(counter, key):
    """Philox4x64-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel random
    numbers: as easy as 1, 2, 3", SC 2011): ten rounds of two 64x64->128-bit products with the
    key bumped by the Weyl constants between rounds. Exact integer arithmetic."""
    c = [int(v) & _U64 for v in counter]
    k0, k1 = int(key[0]) & _U64, int(key[1]) & _U64
    for _ in range(10):
        p0 = _PHILOX_M[0] * c[0]
        p1 = _PHILOX_M[1] * c[2]
        c = [((p1 >> 64) ^ c[1] ^ k0) & _U64, p1 & _U64, ((p0 >> 64) ^ c[3] ^ k1) & _U64, p0 & _U64]
        k0 = (k0 + _PHILOX_W[0]) & _U64
        k1 = (k1 + _PHILOX_W[1]) & _U64
    return c


def routing_noise(T, E, seed):
    """Standard normal noise for every (token t, expert e), four experts per generator draw:
    experts 4g .. 4g+3 of token t take Philox4x64-10 at counter (t, g, 0, 0) with key
    (seed, 0). The top 24 bits of outputs 0, 1 and of outputs 2, 3 give two pairs (u1, u2) in
    (0, 1]; Box-Muller makes each pair the two normals sqrt(-2 ln u1) cos(2 pi u2) and
    sqrt(-2 ln u1) sin(2 pi u2), in that order."""
    n = np.zeros((T, E))
    for t in range(T):
        for g in range((E + 3) // 4):
            o = philox4x64_10((t, g, 0, 0), (seed, 0))
            z = []
            for h in range(2):
                u1 = ((o[2 * h] >> 40) + 1) / float(1 << 24)
                u2 = ((o[2 * h + 1] >> 40) + 1) / float(1 << 24)
                r = math.sqrt(-2.0 * math.log(u1))
                z += [r * math.cos(2.0 * math.pi * u2), r * math.sin(2.0 * math.pi * u2)]
            for j in range(4):
                if 4 * g + j < E:
                    n[t, 4 * g + j] = z[j]
    return n


def route(x, Wg, bg, k, temperature=1.0, noise_std=0.0, noise_seed=0, idx=None):
    """Gate linear, top-k, softmax over the k, counts and balance loss. With noise_std > 0 the
    logits get noise_std * N(0,1) before the selection and the softmax (training-time routing
    noise, PyTorch-MoE page, section 4.3: logits + randn_like(logits) * 0.1); the noise is a
    constant for the backward.

    `idx` [T,k] (optional) replaces the top-k selection with a given one; everything after the
    selection (weights over the selected logits, counts, balance loss) follows from it as
    usual. A token whose neighbouring logits nearly tie has more than one correct selection
    under rounding; this lets the rest of the layer be evaluated on either."""
    z = gate_logits(x, Wg, bg)
    if noise_std > 0:
        z = z + noise_std * routing_noise(z.shape[0], z.shape[1], noise_seed)
    if k == z.shape[1]:
        idx_d, z_sel, gap = select_all(z)
    else:
        idx_d, z_sel = select_topk(z, k)
        gap = topk_gap(z, k)
    if idx is None:
        idx = idx_d
    else:
        idx = np.asarray(idx, dtype=np.int64).reshape(z.shape[0], k)
        z_sel = np.take_along_axis(z, idx, axis=1)
    w = routing_weights(z_sel, temperature)
    counts = expert_counts(idx, z.shape[1])
    return dict(z=z, idx=idx, z_sel=z_sel, w=w, gap=gap, counts=counts,
                balance_loss=balance_loss(counts))


# ----------------------------------------------------------------------------- dispatch

def capacity(capacity_factor, T, k, E):
    """Expert capacity C = ceil(capacity_factor * T * k / E) (PithTrain page 4.3 item 1, with
    tokens_per_batch read as the T*k routed assignments); None means no limit. The product is
    evaluated in double from the fp32 value of the factor, left to right."""
    if capacity_factor is None or capacity_factor <= 0:
        return None
    cf = float(np.float32(capacity_factor))
    return int(math.ceil(cf * float(T) * float(k) / float(E)))


def dispatch(idx, E, C=None, align=1):
    """Stable counting sort of the (token, slot) assignments by expert, with capacity drops.

    Walks tokens in order (slots in order within a token); an assignment to expert e gets
    rank = number of earlier assignments to e and is kept iff rank < C. Kept rows of expert e
    are laid out contiguously in token order inside e's bucket (Expert-Parallelism page 4.2,
    idea 2: tokens written straight to per-expert bucket offsets). Each bucket is padded to a
    multiple of `align` rows (align=1: the dense layout).

    Returns dict: counts [E], kept [E], offsets [E+1] (bucket starts), row_token [offsets[E]]
    (token of each row, -1 on padding), slot_row [T,k] (row of each assignment, -1 dropped),
    rank [T,k], n_dropped.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    seen = np.zeros(E, dtype=np.int64)
    rank = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            rank[t, j] = seen[e]
            seen[e] += 1
    counts = seen.copy()
    kept = counts.copy() if C is None else np.minimum(counts, C)
    padded = -(-kept // align) * align
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    keep = np.ones((T, k), dtype=bool) if C is None else rank < C
    slot_row = np.where(keep, offsets[idx] + rank, -1)
    row_token = np.full(int(offsets[E]), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            if slot_row[t, j] >= 0:
                row_token[slot_row[t, j]] = t
    return dict(counts=counts, kept=kept, offsets=offsets, row_token=row_token,
                slot_row=slot_row, rank=rank, n_dropped=int(T * k - kept.sum()))


def permute(x, row_token):
    """Xp[r] = x[row_token[r]], zero rows where row_token is -1."""
    x = _f64(x)
    Xp = np.zeros((len(row_token), x.shape[1]))
    valid = row_token >= 0
    Xp[valid] = x[row_token[valid]]
    return Xp


# ----------------------------------------------------------------------------- experts

def gelu(a):
    """GELU(a) = a * Phi(a), exact erf form (nn.GELU default; PithTrain page 4.1, PyTorch-MoE 3.2)."""
    a = _f64(a)
    return 0.5 * a * (1.0 + erf(a / math.sqrt(2.0)))


def gelu_prime(a):
    """d GELU / da = Phi(a) + a * phi(a)."""
    a = _f64(a)
    Phi = 0.5 * (1.0 + erf(a / math.sqrt(2.0)))
    phi = np.exp(-0.5 * a * a) / math.sqrt(2.0 * math.pi)
    return Phi + a * phi


def expert_ffn(Xe, W1e, b1e, W2e, b2e):
    """One expert's FFN on its rows: A = X W1^T + b1, H = GELU(A), Y = H W2^T + b2
    (PyTorch-MoE page 3.2, Expert.forward; PithTrain page 4.1 expert_pool)."""
    A = _f64(Xe) @ _f64(W1e).T + _f64(b1e)[None, :]
    H = gelu(A)
    Y = H @ _f64(W2e).T + _f64(b2e)[None, :]
    return A, H, Y


def combine(Yp, w, slot_row, T):
    """y[t] = sum over kept slots j of w[t,j] * Yp[slot_row[t,j]] (PithTrain page 4.1:
    output[mask] += expert_output * routing_weight); a token with every slot dropped gets 0."""
    Yp = _f64(Yp)
    y = np.zeros((T, Yp.shape[1]))
    for j in range(slot_row.shape[1]):
        r = slot_row[:, j]
        ok = r >= 0
        y[ok] += w[ok, j][:, None] * Yp[r[ok]]
    return y


# ----------------------------------------------------------------------------- whole layer

def forward(inp, k, temperature=1.0, C=None, align=1, noise_std=0.0, noise_seed=0, idx=None):
    """Forward of the layer. `inp` holds x, Wg, bg, W1, b1, W2, b2 (any array type); `idx`
    (optional) is a given top-k selection (see route)."""
    x = _f64(inp["x"])
    T = x.shape[0]
    E = np.asarray(inp["Wg"]).shape[0]
    r = route(x, inp["Wg"], inp.get("bg"), k, temperature, noise_std, noise_seed, idx=idx)
    dsp = dispatch(r["idx"], E, C, align)
    Xp = permute(x, dsp["row_token"])
    f = np.asarray(inp["W1"]).shape[1]
    n_rows = Xp.shape[0]
    A = np.zeros((n_rows, f))
    H = np.zeros((n_rows, f))
    Yp = np.zeros((n_rows, x.shape[1]))
    for e in range(E):
        lo, n = dsp["offsets"][e], dsp["kept"][e]
        if n == 0:
            continue
        A[lo:lo + n], H[lo:lo + n], Yp[lo:lo + n] = expert_ffn(
            Xp[lo:lo + n], inp["W1"][e], inp["b1"][e], inp["W2"][e], inp["b2"][e])
    y = combine(Yp, r["w"], dsp["slot_row"], T)
    out = dict(r)
    out.update(dsp)
    out.update(Xp=Xp, A=A, H=H, Yp=Yp, y=y, temperature=float(temperature))
    return out


def backward(inp, fwd, dy):
    """Gradients of L = sum(y * dy) w.r.t. x, Wg, (bg), W1, b1, W2, b2, and the routing
    weights. The top-k selection and the capacity ranks are piecewise constant; the balance
    loss has zero gradient."""
    x = _f64(inp["x"])
    Wg = _f64(inp["Wg"])
    dy = _f64(dy)
    T, d = x.shape
    E = Wg.shape[0]
    idx, w, slot_row = fwd["idx"], fwd["w"], fwd["slot_row"]
    Yp, A, H, Xp = fwd["Yp"], fwd["A"], fwd["H"], fwd["Xp"]
    k = idx.shape[1]
    f = A.shape[1]

    # combine backward: dw[t,j] = <dy[t], Yp[row]>, dYp[row] = w[t,j] dy[t]
    dw = np.zeros((T, k))
    dYp = np.zeros_like(Yp)
    for j in range(k):
        r = slot_row[:, j]
        ok = r >= 0
        dw[ok, j] = np.einsum("td,td->t", dy[ok], Yp[r[ok]])
        dYp[r[ok]] = w[ok, j][:, None] * dy[ok]

    # experts backward
    dW1 = np.zeros((E, f, d))
    db1 = np.zeros((E, f))
    dW2 = np.zeros((E, d, f))
    db2 = np.zeros((E, d))
    dA = np.zeros_like(A)
    dXp = np.zeros_like(Xp)
    for e in range(E):
        lo, n = fwd["offsets"][e], fwd["kept"][e]
        if n == 0:
            continue
        sl = slice(lo, lo + n)
        W1e, W2e = _f64(inp["W1"][e]), _f64(inp["W2"][e])
        dH = dYp[sl] @ W2e
        dA[sl] = dH * gelu_prime(A[sl])
        dW2[e] = dYp[sl].T @ H[sl]
        db2[e] = dYp[sl].sum(axis=0)
        dW1[e] = dA[sl].T @ Xp[sl]
        db1[e] = dA[sl].sum(axis=0)
        dXp[sl] = dA[sl] @ W1e

    # router backward: softmax Jacobian over the k selected, divided by the temperature
    s = (w * dw).sum(axis=1, keepdims=True)
    dz_sel = w * (dw - s) / fwd["temperature"]
    dZ = np.zeros((T, E))
    np.put_along_axis(dZ, idx, dz_sel, axis=1)
    dWg = dZ.T @ x
    dbg = dZ.sum(axis=0)

    dx = dZ @ Wg
    for j in range(k):
        r = slot_row[:, j]
        ok = r >= 0
        dx[ok] += dXp[r[ok]]
    return dict(dw=dw, dYp=dYp, dA=dA, dXp=dXp, dW1=dW1, db1=db1, dW2=dW2, db2=db2,
                dz_sel=dz_sel, dZ=dZ, dWg=dWg, dbg=dbg, dx=dx)


def layer_loss(fwd, dy, aux_loss_weight=AUX_LOSS_WEIGHT):
    """Reported loss: sum(y * dy) + aux_loss_weight * balance_loss (PyTorch-MoE page 4.3)."""
    return float(np.sum(fwd["y"] * _f64(dy)) + aux_loss_weight * fwd["balance_loss"])


# ----------------------------------------------------------------------------- dense soft MoE

def dense_soft_moe(inp, temperature=1.0):
    """Naive soft MoE: g = softmax(z / temperature) over all E experts and
    y = sum_e g_e expert_e(x) on every token (Expert-Parallelism page 2.2)."""
    x = _f64(inp["x"])
    z = gate_logits(x, inp["Wg"], inp.get("bg"))
    g = routing_weights(z, temperature)
    y = np.zeros_like(x)
    for e in range(z.shape[1]):
        _, _, Ye = expert_ffn(x, inp["W1"][e], inp["b1"][e], inp["W2"][e], inp["b2"][e])
        y += g[:, e:e + 1] * Ye
    return dict(z=z, g=g, y=y)


# ----------------------------------------------------------------------------- co-selection

def coselection(idx, E):
    """Expert co-selection matrix of one batch (Expert-Parallelism page, section 3.2, step 1:
    how often experts i and j are chosen by the same token). The page calls the matrix
    asymmetric, which a plain co-occurrence count is not; the reading taken here: for i != j,
    H[i][j] = number of tokens whose top-k holds i in an earlier slot (a higher logit) than
    j, so H + H^T is the co-occurrence count; H[i][i] = number of tokens that chose i."""
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    Hm = np.zeros((E, E), dtype=np.int64)
    for t in range(T):
        for a in range(k):
            Hm[idx[t, a], idx[t, a]] += 1
            for b in range(a + 1, k):
                Hm[idx[t, a], idx[t, b]] += 1
    return Hm


# ----------------------------------------------------------------------------- soft balance loss

def soft_load(z, temperature=1.0):
    """Differentiable expert load: P_e = sum_t softmax(z_t / temperature)_e over all E experts
    (the gate probabilities of Expert-Parallelism page 2.2, summed over the batch)."""
    p = routing_weights(z, temperature)   # softmax over all columns
    return p, p.sum(axis=0)


def soft_balance_loss(P, weight):
    """weight * mean_e (P_e - mean(P))^2: the PyTorch-MoE page 3.3 balance_loss applied to the
    soft load instead of the integer counts, so that it has a gradient."""
    P = _f64(P)
    return float(weight * np.mean((P - P.mean()) ** 2))


def soft_balance_grad(z, temperature, weight):
    """d soft_balance_loss / d z [T, E]: g_e = weight * 2 (P_e - mean P) / E (the mean term
    drops out since sum_e (P_e - mean P) = 0), then the softmax Jacobian per token,
    dz_te = p_te (g_e - sum_j p_tj g_j) / temperature."""
    p, P = soft_load(z, temperature)
    E = P.shape[0]
    g = weight * 2.0 * (P - P.mean()) / E
    s = (p * g[None, :]).sum(axis=1, keepdims=True)
    return p * (g[None, :] - s) / temperature


# ----------------------------------------------------------------------------- sliding window

def sliding_windows(loads, W):
    """The windows of a sequence of batches (Expert-Parallelism page, section 2.3: the expert
    load statistics are taken over the last 100 batches instead of one batch). `loads` lists
    the soft loads P [E] of successive batches; window i holds batches max(0, i - W + 1) .. i,
    oldest first: the current batch and the W - 1 before it (fewer at the start)."""
    loads = [_f64(P) for P in loads]
    return [np.stack(loads[max(0, i - W + 1):i + 1]) for i in range(len(loads))]


def window_balance_loss(P_window, weight):
    """Balance loss on the window mean: Pbar = mean over the window's batches of the soft load,
    loss = weight * mean_e (Pbar_e - mean(Pbar))^2 (the soft_balance_loss form applied to
    Pbar). Returns (Pbar [E], loss)."""
    Pbar = _f64(P_window).mean(axis=0)
    return Pbar, float(weight * np.mean((Pbar - Pbar.mean()) ** 2))


def window_balance_grad(z, temperature, weight, P_window):
    """d window_balance_loss / d z [T, E] of the current batch (the last row of P_window, whose
    soft load is that of z). Earlier batches are stored statistics, constants here, so the
    gradient reaches only the current batch: dloss/dP_now,e = g_e = weight * 2 (Pbar_e -
    mean Pbar) / (E n) with n the window's batch count (the mean term drops out since
    sum_e (Pbar_e - mean Pbar) = 0), then the softmax Jacobian per token,
    dz_te = p_te (g_e - sum_j p_tj g_j) / temperature."""
    p, _ = soft_load(z, temperature)
    P_window = _f64(P_window)
    n, E = P_window.shape
    Pbar = P_window.mean(axis=0)
    g = weight * 2.0 * (Pbar - Pbar.mean()) / (E * n)
    s = (p * g[None, :]).sum(axis=1, keepdims=True)
    return p * (g[None, :] - s) / temperature
