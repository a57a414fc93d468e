"""Helpers of the parity tests: run the CUDA layer through the C ABI and the fp64 oracle on
the same seeded inputs, and compare them.

Tolerance metric per tensor: max_i |gpu_i - orc_i| / max_i |orc_i| <= 2e-2 (bf16) or
1e-4 (fp32); integer outputs must match exactly. Tokens whose top-(k+1) logits are closer
than 1e-5 in the oracle are left out of the index comparison (the GPU accumulates the
logits in fp32, the oracle in fp64).
"""
import numpy as np
import torch

import synth
from oracle import moe_oracle as O

TOL = {"bf16": 2e-2, "f32": 1e-4}
GAP = 1e-5


def tol(cfg):
    return TOL[cfg.dtype]


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def np_inputs(inp):
    return {k: (None if v is None else f64(v)) for k, v in inp.items()}


def to_dev(inp, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def rel_err(gpu, orc):
    gpu = np.asarray(gpu, dtype=np.float64)
    orc = np.asarray(orc, dtype=np.float64)
    assert gpu.shape == orc.shape, (gpu.shape, orc.shape)
    scale = np.abs(orc).max() if orc.size else 0.0
    if scale == 0.0:
        return float(np.abs(gpu).max()) if gpu.size else 0.0
    return float(np.abs(gpu - orc).max() / scale)


def assert_close(name, gpu, orc, tolerance):
    e = rel_err(gpu, orc)
    assert e <= tolerance, f"{name}: max rel err {e:.3e} > {tolerance:.1e}"
    return e


def assert_loss_close(loss_gpu, fwd, dy, tolerance):
    """The reported loss sum(y * dy) + aux_loss_weight * balance_loss against the oracle's. It
    sums T*d products of random sign, so it is far smaller than its terms (cancellation):
    judged like a tensor of those products, its error is bounded by the tolerance times their
    l2 norm ||y * dy||_2 (the scale of a sum of independently rounded terms), not by the
    tolerance times the cancelled total."""
    ref = O.layer_loss(fwd, dy)
    scale = float(np.linalg.norm(np.asarray(fwd["y"], dtype=np.float64) * np.asarray(dy, dtype=np.float64)))
    err = abs(float(loss_gpu) - ref)
    assert err <= tolerance * max(scale, abs(ref), 1e-30), \
        f"loss {loss_gpu} vs {ref}: |err| {err:.3e} > {tolerance:.1e} x {max(scale, abs(ref)):.3e}"
    return err


def oracle_capacity(cfg):
    return O.capacity(cfg.capacity_factor, cfg.T, cfg.k, cfg.E)


def oracle_run(cfg, npin, dy=None, align=128):
    """Oracle forward (+ backward) with buckets padded to `align` rows (the library's
    cfg.row_align, so that the bucket layouts compare bit for bit)."""
    C = oracle_capacity(cfg)
    fwd = O.forward(npin, cfg.k, cfg.temperature, C, align=align)
    bwd = O.backward(npin, fwd, dy) if dy is not None else None
    return fwd, bwd


def act_dtype(cfg):
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


def dev_i32(a, device="cuda"):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32, device=device)


def dev_act(cfg, a, device="cuda"):
    """Oracle values rounded (nearest even) to the layer's storage dtype, on the device."""
    return torch.as_tensor(np.asarray(a), dtype=torch.float64).to(act_dtype(cfg)).to(device)


def dev_f32(a, device="cuda"):
    return torch.as_tensor(np.asarray(a), dtype=torch.float64).to(torch.float32).to(device)


def nontie_tokens(fwd):
    return fwd["gap"] >= GAP


def valid_selection(z, idx, k, gap=GAP):
    """Per token: `idx` is a correct top-k of the logits z up to rounding of `gap`. Its k ids
    are distinct and in range, and its slot-j logit lies within `gap` of the j-th largest
    logit (slot j holds the j-th largest)."""
    z = np.asarray(z, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    E = z.shape[1]
    in_range = ((idx >= 0) & (idx < E)).all(axis=1)
    safe = np.clip(idx, 0, E - 1)
    distinct = np.array([len(set(r)) == k for r in safe])
    order = -np.sort(-z, axis=1)[:, :k]
    close = (np.abs(np.take_along_axis(z, safe, axis=1) - order) <= gap).all(axis=1)
    return in_range & distinct & close


def oracle_on_gpu_routing(cfg, npin, fwd, gidx, dy=None, align=128, noise_std=0.0, noise_seed=0):
    """Reconcile a GPU selection with the oracle's. Outside near-ties (gap >= GAP) the GPU's
    top-k indices must equal the oracle's. A near-tie token may come out either way under
    rounding; there the GPU's choice must be a correct top-k (valid_selection). Returns the
    oracle's forward (and backward) evaluated on the GPU's selection, so that every
    downstream value is still compared, and the number of tokens that were routed the other
    way."""
    gidx = np.asarray(gidx, dtype=np.int64)
    ok = nontie_tokens(fwd)
    assert (gidx[ok] == fwd["idx"][ok]).all(), \
        f"{(gidx[ok] != fwd['idx'][ok]).any(1).sum()} tokens outside near-ties routed differently"
    flipped = (gidx != fwd["idx"]).any(axis=1)
    n_flipped = int(flipped.sum())
    if n_flipped == 0:
        bwd = O.backward(npin, fwd, dy) if dy is not None else None
        return fwd, bwd, 0
    assert valid_selection(fwd["z"][flipped], gidx[flipped], cfg.k).all(), \
        "a near-tie token's GPU selection is not a top-k of its logits"
    C = oracle_capacity(cfg)
    fwd2 = O.forward(npin, cfg.k, cfg.temperature, C, align=align, noise_std=noise_std,
                     noise_seed=noise_seed, idx=gidx)
    bwd2 = O.backward(npin, fwd2, dy) if dy is not None else None
    return fwd2, bwd2, n_flipped


__all__ = ["synth", "O"]
