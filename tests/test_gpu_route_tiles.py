"""Routing with more 128-token tiles than SMs: the top-k router (k < 8) then runs one CTA per
SM over equal shares of smaller tiles, selecting over one tile while the next one loads, and
the k = 8 router runs several waves of CTAs. Small d and many tokens keep the oracle fast.
Indices are compared bit-exact on every token outside the near-tie set, weights to 1e-4, and
the optional logits output element by element."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

CASES = {
    # one epilogue group (E <= 32), three tiles per CTA
    "tiles-e16-k2": (synth.LayerConfig(name="tiles-e16-k2", T=40000, d=64, E=16, k=2, d_ff=64,
                                       capacity_factor=None), 0.0),
    # four groups, a gate bias and routing noise; two tiles per CTA, the last CTA one
    "tiles-e200-k3-noise": (synth.LayerConfig(name="tiles-e200-k3-noise", T=36000, d=128, E=200, k=3, d_ff=64,
                                              capacity_factor=None, gate_bias="zipf", zipf_s=1.2,
                                              zipf_c=synth.configs.ZIPF_C_E64), 0.1),
    # four tiles per CTA (both accumulators reused twice)
    "tiles-e128-k4": (synth.LayerConfig(name="tiles-e128-k4", T=60000, d=64, E=128, k=4, d_ff=64,
                                        capacity_factor=None), 0.0),
    # the top-8 path in several waves of one-tile CTAs
    "tiles-e64-k8": (synth.LayerConfig(name="tiles-e64-k8", T=40000, d=64, E=64, k=8, d_ff=64,
                                       capacity_factor=None, temperature=0.2), 0.0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_route_many_tiles(name, moe_lib, cuda_device):
    moe = moe_lib
    cfg, noise_std = CASES[name]
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    fwd = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature,
                    noise_std=noise_std, noise_seed=1)
    c = moe.config_from(cfg, noise_std=noise_std, noise_seed=1)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=False)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b, logits=logits)
    moe.get_error()
    # the logits output (bias and noise included): fp32 sums of bf16 products against fp64
    P.assert_close("logits", P.f64(logits), fwd["z"], 1e-5)
    idx = b["idx"].cpu().numpy()
    ok = P.nontie_tokens(fwd)
    assert ok.mean() > 0.99
    assert (idx[ok] == fwd["idx"][ok]).all(), f"{(idx[ok] != fwd['idx'][ok]).any(1).sum()} tokens differ"
    assert P.valid_selection(fwd["z"], idx, cfg.k).all()
    w = b["w"].cpu().double().numpy()
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-5)
    P.assert_close("w", w[ok], fwd["w"][ok], 1e-4)
    counts = b["counts"].cpu().numpy()
    assert (counts == np.bincount(idx.reshape(-1), minlength=cfg.E)).all()
