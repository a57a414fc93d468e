"""Training-time routing noise on the GPU against the oracle: both sides draw the same
Philox4x64-10 / Box-Muller normals per (token, expert), so the noisy top-k indices must
match exactly (outside near-ties) and the weights within tolerance; the whole noisy step
(forward and backward) matches the oracle end to end."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

NOISE = 0.1


@pytest.mark.parametrize("name,seed", [("small-top2-cap1.0", 7), ("small-hybrid-top8", 8),
                                       ("small-max-e256-k8", 9), ("tiny-fp32-fwd", 10),
                                       ("top2-e16-cap1.0", 11)])
def test_noisy_route_matches_oracle(name, seed, moe_lib, cuda_device):
    moe = moe_lib
    cfg = synth.get(name)
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    r = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature, noise_std=NOISE, noise_seed=seed)
    c = moe.config_from(cfg, noise_std=NOISE, noise_seed=seed)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=False)
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b)
    moe.get_error()
    ok = P.nontie_tokens(r)
    idx = b["idx"].cpu().numpy()
    assert (idx[ok] == r["idx"][ok]).all(), f"{(idx[ok] != r['idx'][ok]).any(1).sum()} tokens differ"
    P.assert_close("w", b["w"].cpu().double().numpy()[ok], r["w"][ok], 1e-4)
    # the noise changes the routing of a visible share of tokens
    plain = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature)
    assert (plain["idx"] != r["idx"]).any(axis=1).mean() > 0.01


@pytest.mark.parametrize("name,seed", [("small-dense-e8", 12), ("small-dense-e12-cap0.5", 13)])
def test_noisy_dense_route_matches_oracle(name, seed, moe_lib, cuda_device):
    """Dense routing selects every expert, so the noise moves only the weights."""
    moe = moe_lib
    cfg = synth.get(name)
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    r = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature, noise_std=NOISE, noise_seed=seed)
    c = moe.config_from(cfg, noise_std=NOISE, noise_seed=seed)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=False)
    moe.route(c, dev["x"], dev["Wg"], dev["bg"], b)
    moe.get_error()
    assert (b["idx"].cpu().numpy() == r["idx"]).all()
    w = b["w"].cpu().double().numpy()
    P.assert_close("w", w, r["w"], 1e-4)
    plain = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature)
    assert np.abs(plain["w"] - r["w"]).max() > 1e-2


def test_noisy_step_end_to_end(moe_lib, cuda_device):
    moe = moe_lib
    cfg = synth.get("small-top2-cap1.0")
    inp = synth.make_inputs(cfg)
    npin = P.np_inputs(inp)
    c = moe.config_from(cfg, noise_std=NOISE, noise_seed=21)
    C = P.oracle_capacity(cfg)
    fwd = P.O.forward(npin, cfg.k, cfg.temperature, C, align=c.row_align, noise_std=NOISE, noise_seed=21)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=True)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    # a near-tie token routed the other way: the oracle follows the GPU's (valid) selection
    fwd, bwd, _ = P.oracle_on_gpu_routing(cfg, npin, fwd, b["idx"].cpu().numpy(), npin["dy"],
                                          align=c.row_align, noise_std=NOISE, noise_seed=21)
    assert (b["slot_row"].cpu().numpy() == fwd["slot_row"]).all()
    t = P.tol(cfg)
    P.assert_close("y", P.f64(b["y"]), fwd["y"], t)
    for key in ("dx", "dWg", "dW1", "dW2", "db1", "db2"):
        P.assert_close(key, P.f64(b[key]), bwd[key], t)


def test_zero_noise_is_plain_routing(moe_lib, cuda_device):
    moe = moe_lib
    cfg = synth.get("small-zipf-cap1.25")
    dev = P.to_dev(synth.make_inputs(cfg, with_dy=False))
    out = []
    for c in (moe.config_from(cfg), moe.config_from(cfg, noise_std=0.0, noise_seed=99)):
        b = moe.alloc_buffers(c, backward=False)
        moe.route(c, dev["x"], dev["Wg"], dev["bg"], b)
        out.append((b["idx"].clone(), b["w"].clone()))
    moe.get_error()
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
