"""The differentiable balance loss on the soft expert load against the oracle: the routing
logits moe_route can output, the soft load P and the loss (moe_soft_balance), and the
gradient added into dx, dWg and dbg (moe_soft_balance_backward)."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

WEIGHT = 1e-3


@pytest.mark.parametrize("name", ["small-top2-cap1.0", "small-zipf-cap1.25", "small-max-e256-k8",
                                  "small-fp32-bwd", "small-fp32-ragged", "small-dense-e12-cap0.5",
                                  "small-dense-e40", "top2-e16-cap1.0", "top2-e256-clusters-cap1.0"])
def test_soft_balance_matches_oracle(name, moe_lib, cuda_device):
    moe = moe_lib
    cfg = synth.get(name)
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    c = moe.config_from(cfg)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=False)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
    Pg = torch.empty(cfg.E, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    moe.soft_balance(c, logits, WEIGHT, Pg, loss, b["ws"])
    dx = torch.zeros(cfg.T, cfg.d, dtype=P.act_dtype(cfg), device="cuda")
    dWg = torch.zeros(cfg.E, cfg.d, dtype=torch.float32, device="cuda")
    dbg = torch.zeros(cfg.E, dtype=torch.float32, device="cuda")
    moe.soft_balance_backward(c, logits, Pg, WEIGHT, dev["x"], dev["Wg"], dx, dWg, dbg, b["ws"])
    moe.get_error()

    z = P.O.gate_logits(npin["x"], npin["Wg"], npin["bg"])
    P.assert_close("logits", P.f64(logits), z, 1e-5)
    _, Po = P.O.soft_load(z, cfg.temperature)
    P.assert_close("P", P.f64(Pg), Po, 1e-5)
    # fp32 layers: the benchmark spec's fp32 bar (1e-4) on every value. bf16 layers: the loss and the
    # gate gradients come from fp32 logits and fp32 dz, so they are held to 1e-3, stricter
    # than the bf16 bar; dx is stored in bf16 and gets the bf16 bar.
    t = P.tol(cfg)
    t_gate = t if cfg.dtype == "f32" else 1e-3
    lo = P.O.soft_balance_loss(Po, WEIGHT)
    assert abs(loss.item() - lo) <= t_gate * abs(lo), (loss.item(), lo)
    dZ = P.O.soft_balance_grad(z, cfg.temperature, WEIGHT)
    P.assert_close("dx", P.f64(dx), dZ @ npin["Wg"], t)
    P.assert_close("dWg", P.f64(dWg), dZ.T @ npin["x"], t_gate)
    P.assert_close("dbg", P.f64(dbg), dZ.sum(axis=0), t_gate)


def test_soft_balance_backward_accumulates(moe_lib, cuda_device):
    """The gradient is added to what the buffers already hold."""
    moe = moe_lib
    cfg = synth.get("small-top2-cap1.0")
    c = moe.config_from(cfg)
    dev = P.to_dev(synth.make_inputs(cfg, with_dy=False))
    b = moe.alloc_buffers(c, backward=False)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
    Pg = torch.empty(cfg.E, dtype=torch.float32, device="cuda")
    moe.soft_balance(c, logits, 1.0, Pg, torch.empty(1, device="cuda"), b["ws"])
    outs = []
    for init in (0.0, 1.0):
        dx = torch.full((cfg.T, cfg.d), init, dtype=torch.bfloat16, device="cuda")
        dWg = torch.full((cfg.E, cfg.d), init, dtype=torch.float32, device="cuda")
        moe.soft_balance_backward(c, logits, Pg, 1.0, dev["x"], dev["Wg"], dx, dWg, None, b["ws"])
        outs.append((dx.float(), dWg))
    moe.get_error()
    assert torch.allclose(outs[1][1] - 1.0, outs[0][1], atol=1e-5)
    assert torch.allclose(outs[1][0] - 1.0, outs[0][0], atol=2e-2)
