"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term, a wrong
sign or index, a transposed operand, a wrong tie rule or drop priority) fails it:
hand-worked examples (tests/golden/), closed forms, invariants, special cases that reduce
to another formulation, and brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import moe_oracle as O
from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _rand_inputs(T, d, E, f, seed, bias=False, scale_w=0.3):
    rng = np.random.default_rng(seed)
    inp = dict(x=rng.standard_normal((T, d)), Wg=rng.standard_normal((E, d)) * scale_w,
               bg=(rng.standard_normal(E) * 0.5 if bias else None),
               W1=rng.standard_normal((E, f, d)) * scale_w, b1=rng.standard_normal((E, f)) * 0.1,
               W2=rng.standard_normal((E, d, f)) * scale_w, b2=rng.standard_normal((E, d)) * 0.1)
    return inp


# ------------------------------------------------------------------ hand-worked examples

def test_golden_balance_loss():
    g = _load("balance_loss_hand.json")
    idx = np.array(g["expert_indices"])[:, None]
    counts = O.expert_counts(idx, g["E"])
    assert counts.tolist() == g["load"]
    assert O.balance_loss(counts) == pytest.approx(g["balance_loss"], abs=1e-15)


def test_golden_topk_softmax():
    g = _load("topk_softmax_hand.json")
    for case in g["cases"]:
        idx, zsel = O.select_topk(np.array(case["logits"]), case["k"])
        assert idx.tolist() == case["idx"]
        w = O.routing_weights(zsel, case["temperature"])
        np.testing.assert_allclose(w, case["w"], rtol=1e-14, atol=1e-16)


@pytest.mark.parametrize("layout", ["dense", "align4"])
def test_golden_capacity_dispatch(layout):
    g = _load("capacity_dispatch_hand.json")
    align = 1 if layout == "dense" else 4
    out = O.dispatch(np.array(g["idx"]), g["E"], g["C"], align)
    assert out["counts"].tolist() == g["counts"]
    assert out["kept"].tolist() == g["kept"]
    assert out["n_dropped"] == g["n_dropped"]
    for key in ("offsets", "row_token", "slot_row"):
        assert out[key].tolist() == g[layout][key], key


def test_golden_expert_ffn():
    g = _load("expert_ffn_hand.json")
    A, H, Y = O.expert_ffn(np.array(g["x"]), np.array(g["W1"]), np.array(g["b1"]),
                           np.array(g["W2"]), np.array(g["b2"]))
    np.testing.assert_allclose(A, g["A"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(H, g["H"], rtol=1e-13)
    np.testing.assert_allclose(Y, g["Y"], rtol=1e-13)


# ------------------------------------------------------------------ routing invariants

@pytest.mark.parametrize("k,temp", [(1, 1.0), (2, 1.0), (8, 0.2), (8, 1.0)])
def test_weights_sum_to_one(k, temp):
    inp = _rand_inputs(200, 16, 16, 8, seed=k)
    r = O.route(inp["x"], inp["Wg"], None, k, temp)
    np.testing.assert_allclose(r["w"].sum(axis=1), 1.0, atol=1e-12)
    assert (r["w"] > 0).all()
    # slot j holds the j-th largest logit, so weights are non-increasing along the slots
    assert (np.diff(r["w"], axis=1) <= 1e-15).all()
    assert r["counts"].sum() == 200 * k


def test_topk_matches_bruteforce_sort():
    rng = np.random.default_rng(3)
    z = np.round(rng.standard_normal((300, 12)), 1)  # rounding creates many exact ties
    for k in (1, 2, 5, 12):
        idx, _ = O.select_topk(z, k)
        for t in range(z.shape[0]):
            ref = sorted(range(12), key=lambda e: (-z[t, e], e))[:k]
            assert idx[t].tolist() == ref


def test_top1_equals_argmax_of_full_softmax():
    # PyTorch-MoE page 2.3: softmax over all experts then argmax picks the same expert
    inp = _rand_inputs(500, 32, 16, 8, seed=5)
    r = O.route(inp["x"], inp["Wg"], None, 1, 1.0)
    z = r["z"]
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert (r["idx"][:, 0] == p.argmax(axis=1)).all()
    np.testing.assert_allclose(r["w"], 1.0, atol=0)


def test_gate_bias_shifts_logits():
    inp = _rand_inputs(50, 8, 6, 4, seed=9, bias=True)
    z0 = O.gate_logits(inp["x"], inp["Wg"])
    z1 = O.gate_logits(inp["x"], inp["Wg"], inp["bg"])
    np.testing.assert_allclose(z1 - z0, np.broadcast_to(inp["bg"], z0.shape), atol=1e-12)
    # brute-force logits from the per-element definition
    t, e = 7, 3
    assert z1[t, e] == pytest.approx(sum(inp["x"][t, c] * inp["Wg"][e, c] for c in range(8)) + inp["bg"][e], abs=1e-12)


def test_topk_gap():
    z = np.array([[0.0, 1.0, 1.5, 3.0], [2.0, 2.0, 0.0, -1.0]])
    # k=2: sorted row 0 = 3, 1.5, 1, 0 -> gaps 1.5, 0.5 -> 0.5; row 1 = 2, 2, 0 -> 0
    np.testing.assert_allclose(O.topk_gap(z, 2), [0.5, 0.0])


# ------------------------------------------------------------------ balance loss

def test_balance_loss_closed_forms():
    T, k, E = 96, 2, 8
    # perfect balance: every expert receives T*k/E assignments -> 0
    idx = np.arange(T * k).reshape(T, k) % E
    assert O.balance_loss(O.expert_counts(idx, E)) == 0.0
    # everything to one expert: load = [Tk, 0, ..., 0], mean Tk/E ->
    # ((Tk - Tk/E)^2 + (E-1)(Tk/E)^2) / E = (Tk)^2 (E-1) / E^2
    idx = np.full((T, k), 3)
    assert O.balance_loss(O.expert_counts(idx, E)) == pytest.approx((T * k) ** 2 * (E - 1) / E ** 2, rel=1e-15)


def test_balance_loss_matches_page_snippet_semantics():
    # PyTorch-MoE page 3.3 written with torch ops (scatter_add_ of ones, pow(2).mean())
    rng = np.random.default_rng(11)
    idx = rng.integers(0, 10, size=(400, 2))
    ei = torch.from_numpy(idx.reshape(-1))
    load = torch.zeros(10, dtype=torch.float64).scatter_add_(0, ei, torch.ones_like(ei, dtype=torch.float64))
    ref = (load - load.mean()).pow(2).mean().item()
    assert O.balance_loss(O.expert_counts(idx, 10)) == pytest.approx(ref, rel=1e-14)


# ------------------------------------------------------------------ capacity and dispatch

def test_capacity_formula():
    assert O.capacity(1.0, 8192, 2, 16) == 1024
    assert O.capacity(1.25, 16384, 2, 64) == 640
    assert O.capacity(1.0, 32768, 2, 256) == 256
    assert O.capacity(1.0, 1000, 2, 8) == 250
    assert O.capacity(1.0, 1001, 2, 8) == 251          # ceil(250.25)
    assert O.capacity(0.25, 600, 2, 8) == 38           # ceil(37.5)
    assert O.capacity(None, 10, 2, 4) is None and O.capacity(0.0, 10, 2, 4) is None


def _dispatch_bruteforce(idx, E, C):
    """Independent construction: list each expert's tokens in token order, keep the first C."""
    T, k = idx.shape
    per_e = {e: sorted(t for t in range(T) for j in range(k) if idx[t, j] == e) for e in range(E)}
    kept_tokens = {e: (v if C is None else v[:C]) for e, v in per_e.items()}
    return per_e, kept_tokens


@pytest.mark.parametrize("C", [None, 0, 1, 7, 40])
@pytest.mark.parametrize("align", [1, 8, 128])
def test_dispatch_matches_bruteforce(C, align):
    rng = np.random.default_rng(100 + (C or 0))
    T, k, E = 150, 3, 9
    # distinct experts per token, skewed towards low ids
    p = 1.0 / np.arange(1, E + 1)
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)])
    out = O.dispatch(idx, E, C, align)
    per_e, kept_tokens = _dispatch_bruteforce(idx, E, C)
    assert out["counts"].tolist() == [len(per_e[e]) for e in range(E)]
    assert out["kept"].tolist() == [len(kept_tokens[e]) for e in range(E)]
    assert out["kept"].sum() + out["n_dropped"] == T * k
    off = out["offsets"]
    assert off[0] == 0 and all(off[e] % align == 0 for e in range(E + 1))
    for e in range(E):
        n = out["kept"][e]
        assert off[e + 1] - off[e] == -(-n // align) * align
        assert out["row_token"][off[e]:off[e] + n].tolist() == kept_tokens[e]
        assert (out["row_token"][off[e] + n:off[e + 1]] == -1).all()
    # slot_row points at the row that holds the token, and only kept assignments have one
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = out["slot_row"][t, j]
            if t in kept_tokens[e]:
                assert r == off[e] + kept_tokens[e].index(t)
                assert out["row_token"][r] == t
            else:
                assert r == -1
    rows = out["slot_row"][out["slot_row"] >= 0]
    assert len(set(rows.tolist())) == len(rows)  # injective


def test_permute_and_combine_small():
    x = np.arange(12.0).reshape(4, 3)
    row_token = np.array([2, 0, -1, 3])
    Xp = O.permute(x, row_token)
    np.testing.assert_array_equal(Xp, [x[2], x[0], [0, 0, 0], x[3]])
    slot_row = np.array([[1, -1], [-1, -1], [0, 3], [3, 1]])
    w = np.array([[0.6, 0.4], [0.5, 0.5], [0.9, 0.1], [0.7, 0.3]])
    y = O.combine(Xp, w, slot_row, 4)
    np.testing.assert_allclose(y[0], 0.6 * x[0])
    np.testing.assert_allclose(y[1], 0.0)       # every slot dropped -> 0
    np.testing.assert_allclose(y[2], 0.9 * x[2] + 0.1 * x[3])
    np.testing.assert_allclose(y[3], 0.7 * x[3] + 0.3 * x[0])


# ------------------------------------------------------------------ GELU

def test_gelu_identities_and_table_values():
    a = np.linspace(-6, 6, 241)
    np.testing.assert_allclose(O.gelu(a) - O.gelu(-a), a, atol=1e-14)   # x*Phi(x) + x*Phi(-x) = x
    assert O.gelu(np.array(0.0)) == 0.0
    # standard normal table: Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208
    assert O.gelu(np.array(1.0)) == pytest.approx(0.8413447460685429, rel=1e-15)
    assert O.gelu(np.array(2.0)) == pytest.approx(2 * 0.9772498680518208, rel=1e-15)
    assert O.gelu(np.array(-8.0)) == pytest.approx(0.0, abs=1e-13)


def test_gelu_prime_matches_finite_difference():
    a = np.linspace(-5, 5, 101)
    h = 1e-5
    fd = (O.gelu(a + h) - O.gelu(a - h)) / (2 * h)
    np.testing.assert_allclose(O.gelu_prime(a), fd, atol=1e-9)


# ------------------------------------------------------------------ whole layer

def _dense_then_mask(inp, k, temp, C):
    """Brute force: compute every expert on every token, then weight with a dense [T,E]
    matrix that is zero off the kept selections (capacity decided by the brute-force sort)."""
    x = inp["x"]
    T = x.shape[0]
    E = inp["Wg"].shape[0]
    z = x @ inp["Wg"].T + (0 if inp["bg"] is None else inp["bg"][None, :])
    G = np.zeros((T, E))
    idx = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        sel = sorted(range(E), key=lambda e: (-z[t, e], e))[:k]
        idx[t] = sel
        s = np.array([z[t, e] for e in sel]) / temp
        p = np.exp(s - s.max())
        p /= p.sum()
        for j, e in enumerate(sel):
            G[t, e] = p[j]
    _, kept_tokens = _dispatch_bruteforce(idx, E, C)
    mask = np.zeros((T, E), dtype=bool)
    for e, toks in kept_tokens.items():
        mask[toks, e] = True
    G = np.where(mask, G, 0.0)
    y = np.zeros_like(x)
    for e in range(E):
        Ye = O.gelu(x @ inp["W1"][e].T + inp["b1"][e]) @ inp["W2"][e].T + inp["b2"][e]
        y += G[:, e:e + 1] * Ye
    return y


@pytest.mark.parametrize("k,temp,C,bias", [(2, 1.0, None, False), (2, 1.0, 5, False),
                                           (1, 1.0, 6, True), (4, 0.2, None, False),
                                           (4, 0.2, 3, True), (8, 0.5, None, False)])
def test_sparse_equals_dense_bruteforce(k, temp, C, bias):
    inp = _rand_inputs(40, 6, 8, 5, seed=20 + k, bias=bias)
    out = O.forward(inp, k, temp, C, align=4)
    np.testing.assert_allclose(out["y"], _dense_then_mask(inp, k, temp, C), rtol=0, atol=1e-12)


def test_hybrid_k_equals_E_is_dense_soft_moe():
    # selecting all E experts and soft-weighting them is the naive soft MoE of
    # Expert-Parallelism page 2.2
    inp = _rand_inputs(30, 5, 6, 4, seed=31)
    for temp in (0.2, 1.0, 3.0):
        out = O.forward(inp, 6, temp)
        np.testing.assert_allclose(out["y"], O.dense_soft_moe(inp, temp)["y"], atol=1e-12)


def test_golden_dense_soft_routing():
    g = _load("dense_soft_routing_hand.json")
    for case in g["cases"]:
        z = np.array(case["logits"])
        E = z.shape[1]
        r = O.route(z, np.eye(E), None, E, case["temperature"])
        assert r["idx"].tolist() == case["idx"]
        np.testing.assert_allclose(r["w"], case["w"], rtol=1e-14, atol=1e-16)
        assert r["counts"].tolist() == [z.shape[0]] * E
        assert r["balance_loss"] == 0.0


def test_dense_weights_are_the_full_topk_weights_reordered():
    """k = E keeps slot j = expert j; the weight of each expert equals the one the sorted
    top-E selection gives it."""
    rng = np.random.default_rng(71)
    z = rng.standard_normal((50, 7))
    dense = O.route(z, np.eye(7), None, 7, 0.3)
    idx, zsel = O.select_topk(z, 7)
    wt = O.routing_weights(zsel, 0.3)
    back = np.zeros_like(wt)
    np.put_along_axis(back, idx, wt, axis=1)
    np.testing.assert_allclose(dense["w"], back, rtol=0, atol=1e-15)
    assert np.isinf(dense["gap"]).all()


@pytest.mark.parametrize("C,align", [(None, 1), (None, 8), (9, 4), (0, 4), (40, 8)])
def test_dense_dispatch_closed_form(C, align):
    """Every expert receives every token in token order: kept = min(T, C), bucket e starts at
    e * ceil(kept / align) * align, and slot (t, j) sits at row start_j + t when t < kept."""
    T, E = 23, 5
    idx = np.broadcast_to(np.arange(E), (T, E))
    out = O.dispatch(idx, E, C, align)
    kept = T if C is None else min(T, C)
    B = -(-kept // align) * align
    assert out["kept"].tolist() == [kept] * E
    assert out["offsets"].tolist() == [e * B for e in range(E + 1)]
    assert out["n_dropped"] == E * (T - kept)
    for t in range(T):
        for j in range(E):
            assert out["slot_row"][t, j] == (j * B + t if t < kept else -1)
    rt = out["row_token"]
    for e in range(E):
        assert rt[e * B:e * B + kept].tolist() == list(range(kept))
        assert (rt[e * B + kept:(e + 1) * B] == -1).all()


def test_dense_with_capacity_keeps_the_first_tokens():
    """With capacity C < T every expert keeps tokens 0..C-1: those tokens get the naive soft
    MoE output, the rest get 0."""
    inp = _rand_inputs(12, 4, 3, 5, seed=33, bias=True)
    out = O.forward(inp, 3, 0.5, C=5, align=4)
    ref = O.dense_soft_moe(inp, 0.5)["y"]
    np.testing.assert_allclose(out["y"][:5], ref[:5], atol=1e-12)
    assert (out["y"][5:] == 0).all()


def test_temperature_to_zero_approaches_hard_top1():
    inp = _rand_inputs(60, 8, 8, 6, seed=41)
    k = 4
    hard = O.forward(inp, 1, 1.0)  # hard top-1 layer (weight 1 on the best expert)
    errs_w, errs_y = [], []
    for temp in (1.0, 0.1, 0.01, 1e-3):
        out = O.forward(inp, k, temp)
        onehot = np.zeros_like(out["w"])
        onehot[:, 0] = 1.0
        errs_w.append(np.abs(out["w"] - onehot).max())
        errs_y.append(np.abs(out["y"] - hard["y"]).max())
    assert all(a > b for a, b in zip(errs_w, errs_w[1:]))
    assert all(a > b for a, b in zip(errs_y, errs_y[1:]))
    gap = O.topk_gap(hard["z"], 1)
    ok = gap > 0.02
    out = O.forward(inp, k, 1e-3)
    rel = np.abs(out["y"][ok] - hard["y"][ok]).max() / np.abs(hard["y"][ok]).max()
    assert rel < 1e-6


def test_page1_masked_loop_restatement():
    """The PithTrain page 4.1 forward written with torch masks (every expert, boolean mask of
    tokens that chose it, weighted accumulate) agrees with the oracle when there is no capacity."""
    inp = _rand_inputs(64, 8, 6, 12, seed=51)
    x = torch.from_numpy(inp["x"])
    logits = x @ torch.from_numpy(inp["Wg"]).T
    vals, sel = torch.topk(logits, k=2, dim=-1)
    rw = torch.softmax(vals, dim=-1)
    out = torch.zeros_like(x)
    for e in range(6):
        hit = sel == e
        mask = hit.any(dim=-1)
        if mask.any():
            h = torch.nn.functional.gelu(x[mask] @ torch.from_numpy(inp["W1"][e]).T + torch.from_numpy(inp["b1"][e]))
            ye = h @ torch.from_numpy(inp["W2"][e]).T + torch.from_numpy(inp["b2"][e])
            out[mask] += ye * rw[mask][hit[mask]].unsqueeze(-1)
    np.testing.assert_allclose(O.forward(inp, 2)["y"], out.numpy(), atol=1e-12)


def test_layer_loss_includes_balance_term():
    inp = _rand_inputs(20, 4, 4, 3, seed=61)
    out = O.forward(inp, 2)
    dy = np.ones((20, 4))
    assert O.layer_loss(out, dy) == pytest.approx(out["y"].sum() + 0.01 * out["balance_loss"], rel=1e-14)


def test_zipf_calibration_reaches_forty_percent():
    """The skewed workload's gate bias puts expert 0 into about 40% of tokens' top-2
    (Expert-Parallelism page 2.1); checked on a fresh 4096-token draw of the same recipe."""
    cfg = synth.get("top2-e64-zipf-cap1.25").with_(T=4096, backward=False)
    inp = synth.make_inputs(cfg)
    r = O.route(inp["x"].double().numpy(), inp["Wg"].double().numpy(), inp["bg"].double().numpy(), 2)
    share = (r["idx"] == 0).any(axis=1).mean()
    assert 0.37 < share < 0.43


# ------------------------------------------------------------------ co-selection matrix

def test_golden_coselection():
    g = _load("coselection_hand.json")
    assert O.coselection(np.array(g["idx"]), g["E"]).tolist() == g["H"]


def test_coselection_against_one_hot_products():
    """H + H^T off the diagonal equals A^T A of the one-hot selection matrix A [T, E]; the
    diagonal is the per-expert count; slot order decides which triangle a pair lands in."""
    rng = np.random.default_rng(77)
    T, E, k = 300, 10, 4
    z = rng.standard_normal((T, E))
    idx, _ = O.select_topk(z, k)
    Hm = O.coselection(idx, E)
    A = np.zeros((T, E), dtype=np.int64)
    np.put_along_axis(A, idx, 1, axis=1)
    co = A.T @ A
    off = ~np.eye(E, dtype=bool)
    assert (np.diag(Hm) == O.expert_counts(idx, E)).all()
    assert ((Hm + Hm.T)[off] == co[off]).all()
    # i before j in the slots means z_i > z_j: brute force over the logits
    ref = np.zeros((E, E), dtype=np.int64)
    for t in range(T):
        sel = set(idx[t].tolist())
        for i in sel:
            for j in sel:
                if i != j and (z[t, i] > z[t, j] or (z[t, i] == z[t, j] and i < j)):
                    ref[i, j] += 1
    assert (Hm[off] == ref[off]).all()
    # each chosen expert pairs with the k-1 others of its token
    assert ((Hm + Hm.T).sum(axis=1) - 2 * np.diag(Hm) == np.diag(Hm) * (k - 1)).all()
    assert (O.coselection(idx[:, :1], E)[off] == 0).all()


# ------------------------------------------------------------------ routing noise

def test_philox_matches_numpy_bit_generator():
    """The oracle's Philox4x64-10 against numpy's Philox bit generator (same published
    algorithm; numpy advances its counter by one before each block of four outputs)."""
    for ctr, key in [((0, 0, 0, 0), (0, 0)), ((5, 7, 0, 0), (11, 13)),
                     ((2**62 + 3, 3, 2**61, 9), (2**63 - 5, 42)), ((123456, 255, 0, 0), (987654321, 0))]:
        bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
        ref = [int(v) for v in bg.random_raw(4)]
        nxt = [ctr[0] + 1] + list(ctr[1:])
        assert O.philox4x64_10(nxt, key) == ref


def test_routing_noise_is_standard_normal():
    n = O.routing_noise(400, 250, seed=3).reshape(-1)
    assert abs(n.mean()) < 0.01
    assert abs(n.std() - 1.0) < 0.01
    assert abs(((n - n.mean()) ** 4).mean() / n.var() ** 2 - 3.0) < 0.1   # kurtosis of a normal
    assert abs((n > 1.0).mean() - 0.15865525393145707) < 0.004           # 1 - Phi(1)
    # different seeds and different (t, e) give different draws
    assert not np.array_equal(O.routing_noise(3, 4, 1), O.routing_noise(3, 4, 2))


def test_routing_noise_pairs_are_independent():
    """Four experts share one generator draw: the cosine and sine normals of a Box-Muller pair,
    and the two pairs of a draw, are uncorrelated (a reused output would not be),
    and every expert column is N(0, 1) on its own. A ragged last group (E = 10) is filled."""
    n = O.routing_noise(4000, 10, seed=11)
    c = np.corrcoef(n.T)
    off = c[~np.eye(10, dtype=bool)]
    assert np.abs(off).max() < 0.06                      # 4000 samples: sd of r is ~0.016
    assert np.abs(n.mean(axis=0)).max() < 0.06
    assert np.abs(n.std(axis=0) - 1.0).max() < 0.05
    assert len(np.unique(n)) == n.size


def test_noisy_route_is_plain_route_of_noisy_logits():
    inp = _rand_inputs(50, 8, 12, 4, seed=91)
    noisy = O.route(inp["x"], inp["Wg"], None, 2, 1.0, noise_std=0.1, noise_seed=5)
    zn = O.gate_logits(inp["x"], inp["Wg"]) + 0.1 * O.routing_noise(50, 12, 5)
    idx, zsel = O.select_topk(zn, 2)
    assert (noisy["idx"] == idx).all()
    np.testing.assert_allclose(noisy["w"], O.routing_weights(zsel), atol=1e-15)
    plain = O.route(inp["x"], inp["Wg"], None, 2, 1.0, noise_std=0.0, noise_seed=5)
    assert (plain["idx"] == O.select_topk(O.gate_logits(inp["x"], inp["Wg"]), 2)[0]).all()


# ------------------------------------------------------------------ a given selection

def test_given_selection_reproduces_the_oracle_selection():
    """forward(idx = its own selection) is the same computation, value for value."""
    inp = _rand_inputs(60, 12, 6, 10, seed=31)
    C = O.capacity(1.0, 60, 2, 6)
    a = O.forward(inp, 2, 0.7, C, align=4)
    b = O.forward(inp, 2, 0.7, C, align=4, idx=a["idx"])
    for key in ("idx", "w", "counts", "kept", "offsets", "slot_row", "row_token", "y"):
        assert np.array_equal(a[key], b[key]), key
    assert a["balance_loss"] == b["balance_loss"]


def test_given_selection_on_an_exact_tie():
    """Two experts with equal logits: either order is a correct top-2. The oracle's own
    selection takes the lower id first; given the other order, the weights, counts and the
    layout follow that order. Hand-worked: logits (1, 3, 3, 0), temperature 1, so both
    selected weights are 1/2 whichever expert takes slot 0."""
    x = np.array([[1.0, 0.0], [0.0, 1.0]])
    Wg = np.array([[1.0, 0.0], [3.0, 3.0], [3.0, 3.0], [0.0, 0.0]])
    z = O.gate_logits(x, Wg)
    np.testing.assert_array_equal(z[0], [1.0, 3.0, 3.0, 0.0])
    r_own = O.route(x, Wg, None, 2)
    assert r_own["idx"][0].tolist() == [1, 2]
    given = r_own["idx"].copy()
    given[0] = [2, 1]
    r = O.route(x, Wg, None, 2, idx=given)
    assert r["idx"][0].tolist() == [2, 1]
    np.testing.assert_allclose(r["w"][0], [0.5, 0.5], rtol=0, atol=1e-15)
    assert r["counts"].tolist() == r_own["counts"].tolist()
    d = O.dispatch(r["idx"], 4, None, 1)
    # token 0's slot 0 now holds expert 2: its row sits in expert 2's bucket
    assert d["slot_row"][0, 0] == d["offsets"][2]


def test_valid_selection_helper():
    """The parity tests' check that a near-tie token's GPU selection is a correct top-k."""
    import parity as P
    z = np.array([[0.5, 0.2, 0.2 + 5e-6, -1.0],
                  [0.0, 1.0, 2.0, 3.0]])
    # token 0: experts 1 and 2 nearly tie for slot 1; token 1 has no tie
    assert P.valid_selection(z, [[0, 2], [3, 2]], 2).tolist() == [True, True]
    assert P.valid_selection(z, [[0, 1], [3, 2]], 2).tolist() == [True, True]   # within the gap
    assert P.valid_selection(z, [[0, 3], [2, 3]], 2).tolist() == [False, False]  # not the top-2
    assert P.valid_selection(z, [[0, 0], [3, 3]], 2).tolist() == [False, False]  # repeated id
    assert P.valid_selection(z, [[0, 4], [3, -1]], 2).tolist() == [False, False]  # out of range
    assert P.valid_selection(z, [[2, 0], [2, 3]], 2).tolist() == [False, False]  # slot order


# ------------------------------------------------------------------ sliding-window balance loss

def test_golden_sliding_window_balance():
    g = _load("sliding_window_balance_hand.json")
    wins = O.sliding_windows(g["loads"], g["W"])
    assert [w.tolist() for w in wins] == g["windows"]
    for win, Pbar, loss, gexp in zip(wins, g["Pbar"], g["loss"], g["g"]):
        Pb, lo = O.window_balance_loss(win, g["weight"])
        np.testing.assert_allclose(Pb, Pbar, rtol=0, atol=1e-15)
        assert lo == pytest.approx(loss, abs=1e-15)
        # dloss / dP_now (the window's last row) by central differences: g_e = w 2 (Pbar_e - m) / (E n)
        h = 1e-4
        num = []
        for e in range(len(Pbar)):
            up, dn = win.copy(), win.copy()
            up[-1, e] += h
            dn[-1, e] -= h
            num.append((O.window_balance_loss(up, g["weight"])[1] - O.window_balance_loss(dn, g["weight"])[1]) / (2 * h))
        np.testing.assert_allclose(num, gexp, rtol=0, atol=1e-12)


def test_window_before_it_fills_holds_every_batch():
    """With the page's window of 100 batches, the first batches average all batches so far."""
    rng = np.random.default_rng(3)
    loads = [rng.random(6) * 10 for _ in range(5)]
    for i, win in enumerate(O.sliding_windows(loads, 100)):
        assert win.shape == (i + 1, 6)
        np.testing.assert_array_equal(win, np.stack(loads[:i + 1]))
    # and a full ring keeps only the last W, oldest first
    wins = O.sliding_windows(loads, 2)
    np.testing.assert_array_equal(wins[4], np.stack([loads[3], loads[4]]))
