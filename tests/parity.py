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


__all__ = ["synth", "O"]
