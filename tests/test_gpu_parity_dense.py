"""Parity of the naive dense soft MoE workload at full size (k = E = 128: every expert on every
token, softmax(z / 0.2) over all 128), on the launch configuration the benchmark times.

The whole layer is 2.1M expert rows; the oracle computes sampled outputs one by one:
routing and the closed-form bucket layout are compared in full (bit-exact integers), the
forward rows, y, dw and dx on sampled tokens (all 128 experts each), the weight and bias
gradients of sampled experts on sampled hidden units (all tokens), and dWg through a
property that holds at any size: with every expert selected, each token's softmax Jacobian
row sums to zero, so sum_e dWg[e] = 0.
"""
import numpy as np
import pytest

import synth
import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

NAME = "dense-soft-e128-temp0.2"


def test_dense_full_size(moe_lib, cuda_device):
    moe = moe_lib
    O = P.O
    cfg = synth.get(NAME)
    assert cfg.k == cfg.E
    inp = synth.make_inputs(cfg)
    rng = np.random.default_rng(4321)
    x = inp["x"].double().numpy()
    Wg = inp["Wg"].double().numpy()
    dy = inp["dy"].double().numpy()
    b1 = inp["b1"].double().numpy()
    b2 = inp["b2"].double().numpy()
    c = moe.config_from(cfg)

    # ---------------- oracle routing and bucket layout (whole batch)
    r = O.route(x, Wg, None, cfg.k, cfg.temperature)
    C = O.capacity(cfg.capacity_factor, cfg.T, cfg.k, cfg.E)
    dsp = O.dispatch(r["idx"], cfg.E, C, align=c.row_align)

    # ---------------- GPU
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=True)
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b)
    moe.get_error()
    assert (b["idx"].cpu().numpy() == r["idx"]).all()
    P.assert_close("w", b["w"].cpu().double().numpy(), r["w"], 1e-4)
    assert (b["counts"].cpu().numpy() == cfg.T).all()
    assert b["balance_loss"].item() == 0.0

    b["w"].copy_(P.dev_f32(r["w"]))
    moe.dispatch(c, b["idx"], dev["x"], b)
    moe.expert_ffn(c, b["Xp"], b["offsets"], dev["W1"], dev["b1"], dev["W2"], dev["b2"], b)
    moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"])
    moe.backward(c, dev["dy"], dev["x"], dev["Wg"], dev["W1"], dev["W2"], b)
    moe.get_error()

    n = int(dsp["offsets"][-1])
    assert dsp["n_dropped"] == 0 and b["n_dropped"].item() == 0
    assert b["kept"].cpu().tolist() == dsp["kept"].tolist()
    assert b["offsets"].cpu().tolist() == dsp["offsets"].tolist()
    assert (b["slot_row"].cpu().numpy() == dsp["slot_row"]).all()
    assert (b["row_token"][:n].cpu().numpy() == dsp["row_token"]).all()

    t = P.tol(cfg)
    # ---------------- sampled tokens: every expert's rows, y, dw, dx
    toks = np.unique(np.concatenate([rng.choice(cfg.T, 4, replace=False), [0, cfg.T - 1]]))
    nt = len(toks)
    w = r["w"][toks]                       # [nt, E]
    y_o = np.zeros((nt, cfg.d))
    dws = np.zeros((nt, cfg.E))
    dxp = np.zeros((nt, cfg.d))
    rows_o = {"Gp": [], "H": [], "Yp": []}
    rows_g = {"Gp": [], "H": [], "Yp": []}
    for e in range(cfg.E):
        W1e = inp["W1"][e].double().numpy()
        W2e = inp["W2"][e].double().numpy()
        A, H, Yr = O.expert_ffn(x[toks], W1e, b1[e], W2e, b2[e])
        rows = dsp["slot_row"][toks, e]
        if e % 16 == 0:
            for key, v in (("Gp", O.gelu_prime(A)), ("H", H), ("Yp", Yr)):
                rows_o[key].append(v)
                rows_g[key].append(P.f64(b[key][rows]))
        y_o += w[:, e:e + 1] * Yr
        dws[:, e] = np.einsum("td,td->t", dy[toks], Yr)
        dA = ((w[:, e:e + 1] * dy[toks]) @ W2e) * O.gelu_prime(A)
        dxp += dA @ W1e
    for key in ("Gp", "H", "Yp"):
        P.assert_close(key, np.concatenate(rows_g[key]), np.concatenate(rows_o[key]), t)
    s = (w * dws).sum(axis=1, keepdims=True)
    dz = w * (dws - s) / cfg.temperature
    dx_o = dxp + dz @ Wg
    P.assert_close("y", P.f64(b["y"][toks]), y_o, t)
    P.assert_close("dw", P.f64(b["dw"][toks]), dws, t)
    P.assert_close("dx", P.f64(b["dx"][toks]), dx_o, t)

    # ---------------- sampled experts: weight and bias gradients on sampled hidden units
    for e in (0, 77):
        W1e = inp["W1"][e].double().numpy()
        W2e = inp["W2"][e].double().numpy()
        I = np.sort(rng.choice(cfg.d_ff, 8, replace=False))
        dYp = r["w"][:, e:e + 1] * dy
        A = x @ W1e[I].T + b1[e, I]
        dA = (dYp @ W2e[:, I]) * O.gelu_prime(A)
        P.assert_close("dW1", P.f64(b["dW1"][e, I]), dA.T @ x, t)
        P.assert_close("db1", P.f64(b["db1"][e, I]), dA.sum(0), t)
        P.assert_close("dW2", P.f64(b["dW2"][e][:, I]), dYp.T @ O.gelu(A), t)
        P.assert_close("db2", P.f64(b["db2"][e]), dYp.sum(0), t)

    # ---------------- gate gradient: the full softmax Jacobian rows sum to zero
    dWg = P.f64(b["dWg"])
    assert np.abs(dWg).max() > 0
    assert np.abs(dWg.sum(axis=0)).max() <= 1e-3 * np.abs(dWg).sum(axis=0).max()
