"""Backward of the oracle pinned by central finite differences in fp64 and by torch autograd.

L = sum(y * dy). Top-k selection and capacity ranks are piecewise constant, so the inputs
are drawn until every token's top-(k+1) logits are separated by more than 1e-2; then a
step of 1e-6 never changes the routing and the finite differences see only the smooth part.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def _inputs(T, d, E, f, k, seed):
    for s in range(seed, seed + 200):
        rng = np.random.default_rng(s)
        inp = dict(x=rng.standard_normal((T, d)), Wg=rng.standard_normal((E, d)) * 0.5,
                   bg=rng.standard_normal(E) * 0.3,
                   W1=rng.standard_normal((E, f, d)) * 0.4, b1=rng.standard_normal((E, f)) * 0.2,
                   W2=rng.standard_normal((E, d, f)) * 0.4, b2=rng.standard_normal((E, d)) * 0.2)
        if O.topk_gap(O.gate_logits(inp["x"], inp["Wg"], inp["bg"]), k).min() > 1e-2:
            return inp, rng.standard_normal((T, d))
    raise RuntimeError("no well-separated draw")


def _loss(inp, dy, k, temp, C):
    return float(np.sum(O.forward(inp, k, temp, C)["y"] * dy))


CASES = [  # T, d, E, f, k, temperature, capacity
    (7, 4, 5, 3, 2, 1.0, 2),
    (6, 3, 6, 4, 3, 0.4, None),
    (8, 3, 4, 2, 1, 1.0, 1),
    (6, 3, 4, 3, 4, 0.5, None),   # dense soft routing (k = E): the full softmax Jacobian
    (7, 3, 3, 2, 3, 1.0, 4),      # dense with capacity: tokens 4.. dropped by every expert
]


@pytest.mark.parametrize("T,d,E,f,k,temp,C", CASES)
def test_backward_matches_central_differences(T, d, E, f, k, temp, C):
    inp, dy = _inputs(T, d, E, f, k, seed=T * 100 + k)
    fwd = O.forward(inp, k, temp, C)
    if C is not None:
        assert fwd["n_dropped"] > 0  # the capacity path is exercised
    g = O.backward(inp, fwd, dy)
    h = 1e-6
    names = {"x": "dx", "Wg": "dWg", "bg": "dbg", "W1": "dW1", "b1": "db1", "W2": "dW2", "b2": "db2"}
    for p, gname in names.items():
        base = inp[p]
        fd = np.zeros_like(base)
        for i in np.ndindex(base.shape):
            orig = base[i]
            base[i] = orig + h
            lp = _loss(inp, dy, k, temp, C)
            base[i] = orig - h
            lm = _loss(inp, dy, k, temp, C)
            base[i] = orig
            fd[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g[gname], fd, atol=2e-7, rtol=1e-6, err_msg=gname)
    # gradient w.r.t. the routing weights themselves: dL/dw[t,j] = <dy[t], Yp[row]>
    w = fwd["w"]
    for t in range(T):
        for j in range(k):
            r = fwd["slot_row"][t, j]
            ref = 0.0 if r < 0 else float(dy[t] @ fwd["Yp"][r])
            assert g["dw"][t, j] == pytest.approx(ref, abs=1e-12)
    assert np.isfinite(w).all()


def test_backward_matches_torch_autograd():
    """Second opinion with a library routine: the same layer in torch fp64 with autograd,
    top-k and capacity mask taken as given."""
    T, d, E, f, k, temp, C = 40, 6, 8, 5, 2, 0.7, 8
    inp, dy = _inputs(T, d, E, f, k, seed=900)
    fwd = O.forward(inp, k, temp, C)
    g = O.backward(inp, fwd, dy)
    tt = {n: torch.tensor(v, requires_grad=True) for n, v in inp.items()}
    z = tt["x"] @ tt["Wg"].T + tt["bg"]
    idx = torch.from_numpy(fwd["idx"])
    w = torch.softmax(torch.gather(z, 1, idx) / temp, dim=1)
    keep = torch.from_numpy(fwd["slot_row"] >= 0)
    y = torch.zeros(T, d, dtype=torch.float64)
    for j in range(k):
        W1 = tt["W1"][idx[:, j]]
        b1 = tt["b1"][idx[:, j]]
        W2 = tt["W2"][idx[:, j]]
        b2 = tt["b2"][idx[:, j]]
        h = torch.nn.functional.gelu(torch.einsum("tfd,td->tf", W1, tt["x"]) + b1)
        ye = torch.einsum("tdf,tf->td", W2, h) + b2
        y = y + torch.where(keep[:, j:j + 1], w[:, j:j + 1] * ye, torch.zeros_like(ye))
    (y * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(fwd["y"], y.detach().numpy(), atol=1e-12)
    for p, gname in {"x": "dx", "Wg": "dWg", "bg": "dbg", "W1": "dW1", "b1": "db1", "W2": "dW2", "b2": "db2"}.items():
        np.testing.assert_allclose(g[gname], tt[p].grad.numpy(), atol=1e-11, err_msg=gname)


def test_soft_balance_gradient_matches_central_differences():
    """The soft balance loss w.r.t. x, Wg and bg through z = x Wg^T + bg."""
    rng = np.random.default_rng(123)
    T, d, E, temp, lam = 9, 4, 6, 0.7, 0.3
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, d)) * 0.5
    bg = rng.standard_normal(E) * 0.2

    def loss(x_, Wg_, bg_):
        _, P = O.soft_load(O.gate_logits(x_, Wg_, bg_), temp)
        return O.soft_balance_loss(P, lam)

    dZ = O.soft_balance_grad(O.gate_logits(x, Wg, bg), temp, lam)
    grads = {"x": dZ @ Wg, "Wg": dZ.T @ x, "bg": dZ.sum(axis=0)}
    h = 1e-6
    for name, arr in (("x", x), ("Wg", Wg), ("bg", bg)):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            o = arr[i]
            arr[i] = o + h
            lp = loss(x, Wg, bg)
            arr[i] = o - h
            lm = loss(x, Wg, bg)
            arr[i] = o
            fd[i] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grads[name], fd, atol=1e-8, rtol=1e-6, err_msg=name)


def test_soft_balance_closed_forms():
    T, E = 12, 4
    z = np.zeros((T, E))                       # uniform probabilities: P_e = T/E, loss 0
    _, P = O.soft_load(z)
    np.testing.assert_allclose(P, T / E)
    assert O.soft_balance_loss(P, 0.5) == 0.0
    np.testing.assert_allclose(O.soft_balance_grad(z, 1.0, 0.5), 0.0, atol=1e-15)
    z = np.full((T, E), -50.0)
    z[:, 2] = 50.0                             # every token certain of expert 2
    _, P = O.soft_load(z)
    np.testing.assert_allclose(P, [0, 0, T, 0], atol=1e-12)
    assert O.soft_balance_loss(P, 1.0) == pytest.approx(T ** 2 * (E - 1) / E ** 2, rel=1e-12)
    # sum over experts of each token's gradient vanishes (softmax Jacobian rows sum to 0)
    rng = np.random.default_rng(4)
    zz = rng.standard_normal((T, E))
    np.testing.assert_allclose(O.soft_balance_grad(zz, 0.5, 2.0).sum(axis=1), 0.0, atol=1e-12)


def test_window_of_one_batch_is_the_soft_balance_loss():
    rng = np.random.default_rng(11)
    z = rng.standard_normal((9, 6))
    _, P = O.soft_load(z, 0.7)
    Pb, lo = O.window_balance_loss(P[None, :], 0.3)
    np.testing.assert_array_equal(Pb, P)
    assert lo == pytest.approx(O.soft_balance_loss(P, 0.3), rel=1e-14)
    np.testing.assert_allclose(O.window_balance_grad(z, 0.7, 0.3, P[None, :]),
                               O.soft_balance_grad(z, 0.7, 0.3), rtol=0, atol=1e-15)


@pytest.mark.parametrize("n_past", [0, 2, 4])
def test_window_balance_gradient_matches_central_differences(n_past):
    """The loss as a function of the current batch's logits, the past batches' loads fixed:
    its central differences equal window_balance_grad (a missing 1/n, a wrong mean or a
    dropped softmax term would fail)."""
    rng = np.random.default_rng(20 + n_past)
    T, E, temp, weight, W = 7, 5, 0.6, 0.9, 3
    z = rng.standard_normal((T, E))
    past = [rng.random(E) * T for _ in range(n_past)]

    def loss_of(zz):
        _, P = O.soft_load(zz, temp)
        win = O.sliding_windows(past + [P], W)[-1]
        return O.window_balance_loss(win, weight)[1]

    _, P = O.soft_load(z, temp)
    win = O.sliding_windows(past + [P], W)[-1]
    assert win.shape[0] == min(n_past + 1, W)
    g = O.window_balance_grad(z, temp, weight, win)
    h = 1e-6
    num = np.zeros_like(z)
    for t in range(T):
        for e in range(E):
            zp, zm = z.copy(), z.copy()
            zp[t, e] += h
            zm[t, e] -= h
            num[t, e] = (loss_of(zp) - loss_of(zm)) / (2 * h)
    np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-9)
