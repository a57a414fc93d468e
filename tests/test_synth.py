"""The seeded input generators: determinism, shapes, dtypes and recipe structure."""
import numpy as np
import torch

import synth


def test_deterministic_and_shapes():
    cfg = synth.get("small-top2-cap1.0")
    a = synth.make_inputs(cfg)
    b = synth.make_inputs(cfg)
    for key in ("x", "Wg", "W1", "b1", "W2", "b2", "dy"):
        assert torch.equal(a[key], b[key]), key
        assert a[key].dtype == torch.bfloat16
    assert a["x"].shape == (cfg.T, cfg.d)
    assert a["Wg"].shape == (cfg.E, cfg.d)
    assert a["W1"].shape == (cfg.E, cfg.d_ff, cfg.d) and a["b1"].shape == (cfg.E, cfg.d_ff)
    assert a["W2"].shape == (cfg.E, cfg.d, cfg.d_ff) and a["b2"].shape == (cfg.E, cfg.d)
    assert a["bg"] is None
    c = synth.make_inputs(cfg, seed=1)
    assert not torch.equal(a["x"], c["x"])


def test_distributions():
    cfg = synth.get("small-top2-cap1.0").with_(T=4000)
    a = synth.make_inputs(cfg)
    assert abs(a["x"].float().std().item() - 1.0) < 0.02
    assert abs(a["W1"].float().std().item() - 0.02) < 0.001
    assert abs(a["dy"].float().mean().item()) < 0.01


def test_clusters_and_zipf_recipes():
    cfg = synth.get("small-clusters-cap1.0")
    a = synth.make_inputs(cfg)
    x = a["x"].float().numpy()
    # 16 clusters with noise 0.1: rounding distances to the nearest other token are small
    d2 = ((x[:200, None, :] - x[None, :200, :]) ** 2).sum(-1)
    np.fill_diagonal(d2, np.inf)
    assert np.median(np.sqrt(d2.min(axis=1))) < 0.2 * np.sqrt(2 * cfg.d)
    z = synth.get("small-zipf-cap1.25")
    bg = synth.make_inputs(z)["bg"].double().numpy()
    p = np.array([(e + 1.0) ** -1.2 for e in range(z.E)])
    np.testing.assert_allclose(bg, z.zipf_c * np.log(p / p.sum()), rtol=1e-6)
    assert a["x"].dtype == torch.bfloat16


def test_fp32_workload_dtype():
    a = synth.make_inputs(synth.get("tiny-fp32-fwd"))
    assert a["x"].dtype == torch.float32 and a["dy"] is None


def test_pair_odd_case_mixes_odd_and_even_buckets():
    """The pair-tile parity case keeps buckets of both parities of 128-row tiles (an odd one ends
    in a 128-row pair tile) and an average bucket of at least 1024 rows (the pair path)."""
    from oracle import moe_oracle as O
    cfg = synth.get("small-pair-odd")
    a = synth.make_inputs(cfg)
    r = O.route(a["x"].double().numpy(), a["Wg"].double().numpy(), None, cfg.k)
    tiles = [-(-int(n) // 128) for n in r["counts"]]
    assert {t % 2 for t in tiles} == {0, 1}
    assert cfg.T * cfg.k >= 1024 * cfg.E
    assert cfg.d > 256 and cfg.d_ff > 256 and cfg.d % 256 and cfg.d_ff % 256
