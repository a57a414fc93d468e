"""The soft balance loss on a sliding window of batches (moe_soft_balance_window and its
backward) against the oracle, over successive batches: each call stores its batch's soft load
in the caller's ring, takes the loss on the window mean, and adds the gradient (through the
current batch only) into dx, dWg and dbg. Window of 3 over 5 batches, so the ring fills and
wraps; the ring starts as NaN, which shows that no slot is read before it is written."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

WEIGHT = 1e-3
W = 3
BATCHES = 5


@pytest.mark.parametrize("name", ["small-top2-cap1.0", "small-fp32-bwd", "small-fp32-ragged",
                                  "small-max-e256-k8", "small-dense-e40", "top2-e16-cap1.0"])
def test_window_matches_oracle_over_batches(name, moe_lib, cuda_device):
    moe = moe_lib
    O = P.O
    cfg = synth.get(name)
    c = moe.config_from(cfg)
    b = moe.alloc_buffers(c, backward=False)
    ring = torch.full((W, cfg.E), float("nan"), dtype=torch.float32, device="cuda")
    state = torch.zeros(2, dtype=torch.int32, device="cuda")
    t = P.tol(cfg)
    t_gate = t if cfg.dtype == "f32" else 1e-3   # fp32 logits and dz in either case
    loads = []
    for i in range(BATCHES):
        inp = synth.make_inputs(cfg, seed=100 + i, with_dy=False)
        npin = P.np_inputs(inp)
        dev = P.to_dev(inp)
        logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
        moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
        Pg = torch.empty(cfg.E, dtype=torch.float32, device="cuda")
        Pbar = torch.empty(cfg.E, dtype=torch.float32, device="cuda")
        loss = torch.empty(1, dtype=torch.float32, device="cuda")
        moe.soft_balance_window(c, logits, WEIGHT, W, ring, state, Pg, Pbar, loss, b["ws"])
        dx = torch.zeros(cfg.T, cfg.d, dtype=P.act_dtype(cfg), device="cuda")
        dWg = torch.zeros(cfg.E, cfg.d, dtype=torch.float32, device="cuda")
        dbg = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
        moe.soft_balance_window_backward(c, logits, Pbar, WEIGHT, state, dev["x"], dev["Wg"], dx, dWg, dbg,
                                         b["ws"])
        moe.get_error()

        assert state.cpu().tolist() == [(i + 1) % W, min(i + 1, W)]
        z = O.gate_logits(npin["x"], npin["Wg"], npin["bg"])
        _, Po = O.soft_load(z, cfg.temperature)
        loads.append(Po)
        win = O.sliding_windows(loads, W)[-1]
        Pbo, lo = O.window_balance_loss(win, WEIGHT)
        P.assert_close("P", P.f64(Pg), Po, 1e-5)
        P.assert_close("Pbar", P.f64(Pbar), Pbo, 1e-5)
        assert np.isfinite(ring.cpu().numpy()[:min(i + 1, W)]).all()
        assert abs(loss.item() - lo) <= t_gate * abs(lo), (i, loss.item(), lo)
        dZ = O.window_balance_grad(z, cfg.temperature, WEIGHT, win)
        P.assert_close("dx", P.f64(dx), dZ @ npin["Wg"], t)
        P.assert_close("dWg", P.f64(dWg), dZ.T @ npin["x"], t_gate)
        P.assert_close("dbg", P.f64(dbg), dZ.sum(axis=0), t_gate)


def test_window_of_one_is_the_soft_balance_loss(moe_lib, cuda_device):
    """W = 1: the window holds only the current batch, so loss and gradient equal those of
    moe_soft_balance / moe_soft_balance_backward (up to the mean of P taken by a reduction
    instead of T/E)."""
    moe = moe_lib
    cfg = synth.get("small-zipf-cap1.25")
    c = moe.config_from(cfg)
    dev = P.to_dev(synth.make_inputs(cfg, with_dy=False))
    b = moe.alloc_buffers(c, backward=False)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
    outs = []
    for window in (False, True):
        Pg = torch.empty(cfg.E, device="cuda")
        loss = torch.empty(1, device="cuda")
        dx = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
        dWg = torch.zeros(cfg.E, cfg.d, device="cuda")
        if window:
            ring = torch.empty(1, cfg.E, device="cuda")
            state = torch.zeros(2, dtype=torch.int32, device="cuda")
            Pbar = torch.empty(cfg.E, device="cuda")
            for _ in range(2):      # a second call replaces the first: the window stays one batch
                moe.soft_balance_window(c, logits, WEIGHT, 1, ring, state, Pg, Pbar, loss, b["ws"])
            moe.soft_balance_window_backward(c, logits, Pbar, WEIGHT, state, dev["x"], dev["Wg"], dx, dWg, None,
                                             b["ws"])
            assert state.cpu().tolist() == [0, 1]
            assert torch.equal(Pbar, Pg)
        else:
            moe.soft_balance(c, logits, WEIGHT, Pg, loss, b["ws"])
            moe.soft_balance_backward(c, logits, Pg, WEIGHT, dev["x"], dev["Wg"], dx, dWg, None, b["ws"])
        outs.append((loss.item(), dx.float(), dWg))
    moe.get_error()
    assert outs[1][0] == pytest.approx(outs[0][0], rel=1e-5)
    assert P.rel_err(outs[1][2].cpu().numpy(), outs[0][2].cpu().numpy()) <= 1e-5
    assert P.rel_err(outs[1][1].cpu().numpy(), outs[0][1].cpu().numpy()) <= 1e-2


def test_window_state_out_of_range_is_reported(moe_lib, cuda_device):
    """A corrupted state (slot beyond the ring) is not used to index the ring: the call records
    MOE_ERR_DEVICE_BOUNDS and restarts the window at slot 0."""
    moe = moe_lib
    cfg = synth.get("small-top2-cap1.0")
    c = moe.config_from(cfg)
    dev = P.to_dev(synth.make_inputs(cfg, with_dy=False))
    b = moe.alloc_buffers(c, backward=False)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
    ring = torch.zeros(W, cfg.E, device="cuda")
    state = torch.tensor([W + 5, 1], dtype=torch.int32, device="cuda")
    Pg, Pbar, loss = torch.empty(cfg.E, device="cuda"), torch.empty(cfg.E, device="cuda"), torch.empty(1, device="cuda")
    moe.soft_balance_window(c, logits, WEIGHT, W, ring, state, Pg, Pbar, loss, b["ws"])
    with pytest.raises(moe.MoeError) as ei:
        moe.get_error()
    assert ei.value.status == moe.MOE_ERR_DEVICE_BOUNDS
    assert state.cpu().tolist() == [1, 1]
    assert torch.equal(Pbar, Pg) and torch.equal(ring[0], Pg)
