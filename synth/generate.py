"""Seeded synthetic inputs for the MoE layer, shared by the oracle side and the CUDA side.

Holds none of the method's arithmetic: it only draws random tensors in a fixed order
from one torch CPU generator and rounds them to the storage dtype (round to nearest
even for bf16). "N(0, s)" means standard deviation s.

Draw order per workload: x, Wg, [bg is deterministic], W1, b1, W2, b2, dy.
Layouts follow nn.Linear: Wg [E, d], W1 [E, d_ff, d], b1 [E, d_ff], W2 [E, d, d_ff], b2 [E, d].

x recipes
* "normal":   x ~ N(0, 1)
* "clusters": n_clusters centres mu_j ~ N(0, 1)^d, token t draws j(t) uniformly, then
              x_t = mu_j(t) + N(0, cluster_noise^2)   (correlated expert co-selection,
              "Expert Parallelism" page, section 3.2)
gate bias recipe
* "zipf":     bg_e = c * ln(p_e), p_e proportional to (e+1)^-s (skewed expert load,
              "Expert Parallelism" page, section 2.1). Kept in fp32.
"""
import torch

from .configs import LayerConfig


def _storage_dtype(cfg: LayerConfig) -> torch.dtype:
    if cfg.dtype == "bf16":
        return torch.bfloat16
    if cfg.dtype == "f32":
        return torch.float32
    raise ValueError(f"unknown dtype {cfg.dtype!r}")


def zipf_gate_bias(E: int, s: float, c: float) -> torch.Tensor:
    p = torch.tensor([(e + 1.0) ** (-s) for e in range(E)], dtype=torch.float64)
    p = p / p.sum()
    return (c * torch.log(p)).to(torch.float32)


def make_inputs(cfg: LayerConfig, seed: int = None, with_dy: bool = None) -> dict:
    """Return a dict of CPU tensors: x, Wg, bg (or None), W1, b1, W2, b2, dy (or None)."""
    seed = cfg.seed if seed is None else seed
    with_dy = cfg.backward if with_dy is None else with_dy
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dt = _storage_dtype(cfg)
    T, d, E, f = cfg.T, cfg.d, cfg.E, cfg.d_ff
    std = cfg.weight_std

    def normal(shape, scale=1.0):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * scale)

    if cfg.x_dist == "normal":
        x = normal((T, d)).to(dt)
    elif cfg.x_dist == "clusters":
        centres = normal((cfg.n_clusters, d))
        which = torch.randint(0, cfg.n_clusters, (T,), generator=g)
        x = (centres[which] + normal((T, d), cfg.cluster_noise)).to(dt)
    else:
        raise ValueError(f"unknown x_dist {cfg.x_dist!r}")

    Wg = normal((E, d), std).to(dt)
    bg = zipf_gate_bias(E, cfg.zipf_s, cfg.zipf_c) if cfg.gate_bias == "zipf" else None
    W1 = normal((E, f, d), std).to(dt)
    b1 = normal((E, f), std).to(dt)
    W2 = normal((E, d, f), std).to(dt)
    b2 = normal((E, d), std).to(dt)
    dy = normal((T, d)).to(dt) if with_dy else None
    return dict(x=x, Wg=Wg, bg=bg, W1=W1, b1=b1, W2=W2, b2=b2, dy=dy)


def input_bytes(cfg: LayerConfig) -> int:
    """Bytes of the tensors make_inputs returns (for sizing host memory)."""
    es = 2 if cfg.dtype == "bf16" else 4
    T, d, E, f = cfg.T, cfg.d, cfg.E, cfg.d_ff
    n = T * d + E * d + 2 * E * f * d + E * f + E * d + (T * d if cfg.backward else 0)
    return n * es + (4 * E if cfg.gate_bias == "zipf" else 0)


__all__ = ["make_inputs", "zipf_gate_bias", "input_bytes"]
