"""Parity at the workloads' full sizes, on the launch configuration the benchmark times.

The oracle cannot run these layers whole in a test, so it computes sampled outputs one by
one: routing and the bucket layout are compared in full (integers, bit-exact), values on a
seeded sample of tokens, rows, hidden units and experts. Each GPU stage is fed the oracle's
routing so that a near-tie token (logit gap < 1e-5) cannot shift other tokens' capacity
ranks; the route stage itself is compared on every token outside the near-tie set.
"""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# the dense soft MoE workload (k = E) has its own full-size test
FULL = [n for n, c in synth.WORKLOADS.items() if c.dtype == "bf16" and c.k < c.E]


def _rows_of(dsp, e):
    lo, n = int(dsp["offsets"][e]), int(dsp["kept"][e])
    return np.arange(lo, lo + n)


@pytest.mark.parametrize("name", FULL)
def test_full_size(name, moe_lib, cuda_device):
    moe = moe_lib
    O = P.O
    cfg = synth.get(name)
    inp = synth.make_inputs(cfg)
    rng = np.random.default_rng(1234)
    x = inp["x"].double().numpy()
    Wg = inp["Wg"].double().numpy()
    bg = None if inp["bg"] is None else inp["bg"].double().numpy()
    dy = inp["dy"].double().numpy()
    b1 = inp["b1"].double().numpy()
    b2 = inp["b2"].double().numpy()
    cache = {}

    def Wf(e):
        """fp64 copies of expert e's weights (a few experts kept at a time)."""
        if e not in cache:
            if len(cache) >= 8:
                cache.pop(next(iter(cache)))
            cache[e] = (inp["W1"][e].double().numpy(), inp["W2"][e].double().numpy())
        return cache[e]

    def expert_rows(pairs):
        """Oracle A, H, Yp of the (token, slot) pairs, computed expert by expert."""
        out = {}
        by_e = {}
        for tk, j in pairs:
            by_e.setdefault(int(r["idx"][tk, j]), []).append((tk, j))
        for e, lst in sorted(by_e.items()):
            W1e, W2e = Wf(e)
            tk = np.array([a for a, _ in lst])
            A, H, Yr = O.expert_ffn(x[tk], W1e, b1[e], W2e, b2[e])
            for i, key in enumerate(lst):
                out[key] = (e, A[i], H[i], Yr[i])
        return out

    # ---------------- oracle routing and bucket layout (whole batch)
    r = O.route(x, Wg, bg, cfg.k, cfg.temperature)
    C = O.capacity(cfg.capacity_factor, cfg.T, cfg.k, cfg.E)
    dsp = O.dispatch(r["idx"], cfg.E, C, align=moe.config_from(cfg).row_align)
    ok = P.nontie_tokens(r)

    # ---------------- GPU, same entry points and launch configuration as the benchmark
    dev = P.to_dev(inp)
    c = moe.config_from(cfg)
    b = moe.alloc_buffers(c, backward=True)
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b)
    moe.get_error()
    gidx = b["idx"].cpu().numpy()
    assert (gidx[ok] == r["idx"][ok]).all(), f"{(gidx[ok] != r['idx'][ok]).any(1).sum()} tokens routed differently"
    gw = b["w"].cpu().double().numpy()
    P.assert_close("w", gw[ok], r["w"][ok], 1e-4)
    assert b["counts"].cpu().numpy().sum() == cfg.T * cfg.k
    if ok.all():
        assert (b["counts"].cpu().numpy() == r["counts"]).all()

    # feed the oracle's routing to the remaining stages
    b["idx"].copy_(P.dev_i32(r["idx"]))
    b["w"].copy_(P.dev_f32(r["w"]))
    moe.dispatch(c, b["idx"], dev["x"], b)
    moe.expert_ffn(c, b["Xp"], b["offsets"], dev["W1"], dev["b1"], dev["W2"], dev["b2"], b)
    moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"])
    moe.backward(c, dev["dy"], dev["x"], dev["Wg"], dev["W1"], dev["W2"], b)
    moe.get_error()

    n = int(dsp["offsets"][-1])
    assert b["kept"].cpu().tolist() == dsp["kept"].tolist()
    assert b["offsets"].cpu().tolist() == dsp["offsets"].tolist()
    assert b["n_dropped"].item() == dsp["n_dropped"]
    assert (b["slot_row"].cpu().numpy() == dsp["slot_row"]).all()
    assert (b["row_token"][:n].cpu().numpy() == dsp["row_token"]).all()

    t = P.tol(cfg)
    # ---------------- sampled tokens: forward rows, y, dw, dx
    toks = np.unique(np.concatenate([rng.choice(cfg.T, 48, replace=False), [0, cfg.T - 1],
                                     np.nonzero((dsp["slot_row"] < 0).any(1))[0][:8]]))
    y_o, y_g, dx_o, dx_g, dw_o, dw_g = [], [], [], [], [], []
    rows_o, rows_g = {"Gp": [], "H": [], "Yp": []}, {"Gp": [], "H": [], "Yp": []}
    fr = expert_rows([(tk, j) for tk in toks for j in range(cfg.k) if dsp["slot_row"][tk, j] >= 0])
    for tk in toks:
        yk = np.zeros(cfg.d)
        dws = np.zeros(cfg.k)
        dxp = np.zeros(cfg.d)
        for j in range(cfg.k):
            row = dsp["slot_row"][tk, j]
            if row < 0:
                continue
            e, A, H, Yr = fr[(tk, j)]
            for key, v in (("Gp", O.gelu_prime(A)), ("H", H), ("Yp", Yr)):
                rows_o[key].append(v)
                rows_g[key].append(P.f64(b[key][row]))
            W1e, W2e = Wf(e)
            yk += r["w"][tk, j] * Yr
            dws[j] = dy[tk] @ Yr
            dA = ((r["w"][tk, j] * dy[tk]) @ W2e) * O.gelu_prime(A)
            dxp += dA @ W1e
        s = (r["w"][tk] * dws).sum()
        dz = r["w"][tk] * (dws - s) / cfg.temperature
        dxk = dxp + dz @ Wg[r["idx"][tk]]
        y_o.append(yk); y_g.append(P.f64(b["y"][tk]))
        dx_o.append(dxk); dx_g.append(P.f64(b["dx"][tk]))
        dw_o.append(dws); dw_g.append(P.f64(b["dw"][tk]))
    for key in ("Gp", "H", "Yp"):
        P.assert_close(key, np.array(rows_g[key]), np.array(rows_o[key]), t)
    P.assert_close("y", np.array(y_g), np.array(y_o), t)
    P.assert_close("dw", np.array(dw_g), np.array(dw_o), t)
    P.assert_close("dx", np.array(dx_g), np.array(dx_o), t)

    # ---------------- sampled experts: weight and bias gradients on sampled hidden units
    busy = np.nonzero(dsp["kept"] > 0)[0]
    experts = np.unique(np.concatenate([rng.choice(busy, min(3, len(busy)), replace=False),
                                        [busy[np.argmax(dsp["kept"][busy])]]]))
    g_dW1, o_dW1, g_dW2, o_dW2, g_db1, o_db1, g_db2, o_db2 = [], [], [], [], [], [], [], []
    for e in experts:
        rows = _rows_of(dsp, e)
        tok = dsp["row_token"][rows]
        slot = np.array([np.nonzero(dsp["slot_row"][tt] == rr)[0][0] for tt, rr in zip(tok, rows)])
        Xe = x[tok]
        dYp = r["w"][tok, slot][:, None] * dy[tok]
        I = np.sort(rng.choice(cfg.d_ff, 8, replace=False))
        W1e, W2e = Wf(e)
        A = Xe @ W1e[I].T + b1[e, I]
        dA = (dYp @ W2e[:, I]) * O.gelu_prime(A)
        o_dW1.append(dA.T @ Xe); g_dW1.append(P.f64(b["dW1"][e, I]))
        o_db1.append(dA.sum(0)); g_db1.append(P.f64(b["db1"][e, I]))
        o_dW2.append(dYp.T @ O.gelu(A)); g_dW2.append(P.f64(b["dW2"][e][:, I]))
        o_db2.append(dYp.sum(0)); g_db2.append(P.f64(b["db2"][e]))
    P.assert_close("dW1", np.array(g_dW1), np.array(o_dW1), t)
    P.assert_close("db1", np.array(g_db1), np.array(o_db1), t)
    P.assert_close("dW2", np.array(g_dW2), np.array(o_dW2), t)
    P.assert_close("db2", np.array(g_db2), np.array(o_db2), t)
    # experts without rows have exactly zero gradients
    empty = torch.as_tensor(np.nonzero(dsp["kept"] == 0)[0], device=b["dW1"].device)
    if empty.numel():
        assert (b["dW1"][empty] == 0).all() and (b["dW2"][empty] == 0).all()

    # ---------------- gate gradient on the least-loaded expert that has assignments
    cand = np.nonzero(r["counts"] > 0)[0]
    e = cand[np.argmin(r["counts"][cand])]
    users = np.nonzero((r["idx"] == e).any(1))[0]
    fr = expert_rows([(tk, j) for tk in users for j in range(cfg.k) if dsp["slot_row"][tk, j] >= 0])
    dwg = np.zeros(cfg.d)
    for tk in users:
        dws = np.zeros(cfg.k)
        for j in range(cfg.k):
            if dsp["slot_row"][tk, j] >= 0:
                dws[j] = dy[tk] @ fr[(tk, j)][3]
        s = (r["w"][tk] * dws).sum()
        jj = int(np.nonzero(r["idx"][tk] == e)[0][0])
        dwg += r["w"][tk, jj] * (dws[jj] - s) / cfg.temperature * x[tk]
    P.assert_close("dWg", P.f64(b["dWg"][e]), dwg, t)
