"""Degenerate batches through the whole layer on the GPU: an empty batch (T = 0), a single
token, a single expert (k = E = 1), and a capacity of one row per expert (almost every
assignment dropped). The empty batch is checked against its closed form; the others against
the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

BASE = synth.LayerConfig(name="degenerate", T=0, d=128, E=8, k=2, d_ff=256, capacity_factor=1.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_batch(dtype, moe_lib, cuda_device):
    """No tokens: every call succeeds, nothing is routed or kept, the balance loss and the
    reported loss are 0, and every weight and bias gradient is exactly zero."""
    moe = moe_lib
    cfg = BASE.with_(dtype=dtype)
    inp = synth.make_inputs(cfg)
    dev = P.to_dev(inp)
    c = moe.config_from(cfg)
    assert c.rows_capacity == 0
    b = moe.alloc_buffers(c, backward=True)
    for key in ("dWg", "dW1", "db1", "dW2", "db2", "balance_loss", "loss"):
        b[key].fill_(7.0)                       # stale values must be overwritten
    b["counts"].fill_(5)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    assert (b["counts"] == 0).all() and (b["kept"] == 0).all() and (b["offsets"] == 0).all()
    assert b["n_dropped"].item() == 0
    assert b["balance_loss"].item() == 0.0 and b["loss"].item() == 0.0
    for key in ("dWg", "dW1", "db1", "dW2", "db2"):
        assert (b[key] == 0).all(), key


CASES = {
    "single-token": BASE.with_(name="single-token", T=1, E=4, k=2),
    "single-token-f32": BASE.with_(name="single-token-f32", T=1, d=40, E=5, k=3, d_ff=24, dtype="f32"),
    "single-expert": BASE.with_(name="single-expert", T=200, E=1, k=1, capacity_factor=None),
    "one-row-per-expert": BASE.with_(name="one-row-per-expert", T=400, E=8, k=2, capacity_factor=0.01),
}


@pytest.mark.parametrize("name", list(CASES))
def test_degenerate_layer_matches_oracle(name, moe_lib, cuda_device):
    moe = moe_lib
    cfg = CASES[name]
    inp = synth.make_inputs(cfg)
    npin = P.np_inputs(inp)
    c = moe.config_from(cfg)
    fwd, bwd = P.oracle_run(cfg, npin, npin["dy"], align=c.row_align)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=True)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    # a near-tie token routed the other way: the oracle follows the GPU's (valid) selection
    fwd, bwd, _ = P.oracle_on_gpu_routing(cfg, npin, fwd, b["idx"].cpu().numpy(), npin["dy"],
                                          align=c.row_align)
    n = int(fwd["offsets"][-1])
    assert b["kept"].cpu().tolist() == fwd["kept"].tolist()
    assert b["offsets"].cpu().tolist() == fwd["offsets"].tolist()
    assert b["n_dropped"].item() == fwd["n_dropped"]
    assert (b["slot_row"].cpu().numpy() == fwd["slot_row"]).all()
    assert (b["row_token"][:n].cpu().numpy() == fwd["row_token"]).all()
    t = P.tol(cfg)
    P.assert_close("y", P.f64(b["y"]), fwd["y"], t)
    for key in ("dx", "dWg", "dW1", "db1", "dW2", "db2", "dw"):
        P.assert_close(key, P.f64(b[key]), bwd[key], t)
    # experts that kept no rows have exactly zero weight gradients
    for e in np.nonzero(fwd["kept"] == 0)[0]:
        assert (b["dW1"][e] == 0).all() and (b["dW2"][e] == 0).all()
