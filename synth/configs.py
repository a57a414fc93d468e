"""Layer configurations of the MoE token-routing workloads.

Plain parameter records, no arithmetic of the method. The five workloads follow the
shapes the pages describe for an MoE layer (tokens x dim activations, num_experts,
top-k, capacity_factor, temperature; expert FFN Linear(d, d_ff) -> GELU -> Linear(d_ff, d)):

* "PithTrain" page, section 4.1 (PithTrainMoELayer: gate Linear(dim, num_experts,
  bias=False), experts nn.Sequential(Linear(dim, 4*dim), GELU, Linear(4*dim, dim)),
  top-2) and section 4.3 (capacity_factor 1.0-1.5).
* "PyTorch distributed MoE" page, section 3.2 (Expert(d_model, d_ff)) and 3.3
  (balance_loss), section 4.3 (aux_loss_weight = 0.01).
* "Expert Parallelism" page, section 2.1 (skewed expert load, top expert ~40% of
  tokens), section 2.2 (temperature 0.2; hybrid top-8 pre-selection then soft
  weighting; the naive soft MoE runs every expert on every token), section 3.2 (expert
  co-selection).

The small cases are scaled-down versions of the same recipes: they span several
128-row tiles, have ragged tails and finish in the oracle within seconds.
"""
from dataclasses import dataclass, field, replace
from typing import Optional


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int                      # tokens in the batch
    d: int                      # model dim
    E: int                      # number of experts
    k: int                      # experts selected per token (k = E: dense soft routing)
    d_ff: int                   # expert hidden dim
    capacity_factor: Optional[float] = None   # None: no capacity limit
    temperature: float = 1.0    # softmax temperature over the k selected logits (all E if k = E)
    dtype: str = "bf16"         # storage dtype of activations and weights: "bf16" or "f32"
    backward: bool = True       # whether the workload includes the backward pass
    x_dist: str = "normal"      # "normal": x ~ N(0,1); "clusters": centre ~ N(0,1) + N(0, noise^2)
    n_clusters: int = 0
    cluster_noise: float = 0.0
    gate_bias: str = "none"     # "none" or "zipf": fixed gate bias c*ln(p_e), p_e ~ (e+1)^-s
    zipf_s: float = 0.0
    zipf_c: float = 0.0
    weight_std: float = 0.02    # std of every weight and bias draw
    aux_loss_weight: float = 0.01
    seed: int = 0

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# Scale of the Zipf gate bias for the 64-expert skewed workload. Chosen so that on the
# seed-0 inputs about 40% of tokens carry expert 0 in their top-2 (the "Expert
# Parallelism" page, section 2.1, reports a top expert picked by ~40% of tokens).
# Found by bisection with oracle/calibrate_zipf_bias.py; the value is an input-recipe
# parameter only.
ZIPF_C_E64 = 0.453125

WORKLOADS = {
    # tiny forward-only fp32 layer (tolerance 1e-4)
    "tiny-fp32-fwd": LayerConfig(
        name="tiny-fp32-fwd", T=256, d=64, E=8, k=2, d_ff=256, capacity_factor=None,
        dtype="f32", backward=False),
    # top-2 over 16 experts, capacity factor 1.0
    "top2-e16-cap1.0": LayerConfig(
        name="top2-e16-cap1.0", T=8192, d=1024, E=16, k=2, d_ff=4096, capacity_factor=1.0),
    # top-2 over 64 experts with a Zipf(1.2) gate bias skewing the load, capacity 1.25
    "top2-e64-zipf-cap1.25": LayerConfig(
        name="top2-e64-zipf-cap1.25", T=16384, d=2048, E=64, k=2, d_ff=4096,
        capacity_factor=1.25, gate_bias="zipf", zipf_s=1.2, zipf_c=ZIPF_C_E64),
    # hybrid soft routing: top-8 pre-selection, softmax(z/0.2) over the 8
    "hybrid-top8-e128-temp0.2": LayerConfig(
        name="hybrid-top8-e128-temp0.2", T=16384, d=1024, E=128, k=8, d_ff=4096,
        capacity_factor=None, temperature=0.2),
    # 256 experts, tokens drawn from 64 clusters so co-selection is correlated
    "top2-e256-clusters-cap1.0": LayerConfig(
        name="top2-e256-clusters-cap1.0", T=32768, d=1024, E=256, k=2, d_ff=2048,
        capacity_factor=1.0, x_dist="clusters", n_clusters=64, cluster_noise=0.1),
    # naive dense soft MoE: the hybrid layer's shapes with every one of the 128 experts run
    # on every token, softmax(z/0.2) over all 128 (k = E)
    "dense-soft-e128-temp0.2": LayerConfig(
        name="dense-soft-e128-temp0.2", T=16384, d=1024, E=128, k=128, d_ff=4096,
        capacity_factor=None, temperature=0.2),
}

# The throughput workload the benchmark times by default: the configuration with the most
# work per step (hybrid top-8 over 128 experts, 131,072 expert rows, ~6.6 TFLOP fwd+bwd).
HEADLINE = "hybrid-top8-e128-temp0.2"

# Scaled-down parity cases: several 128-row tiles, ragged tails, drops, skew.
SMALL_CASES = {
    "small-top2-cap1.0": LayerConfig(
        name="small-top2-cap1.0", T=1000, d=256, E=8, k=2, d_ff=512, capacity_factor=1.0),
    "small-zipf-cap1.25": LayerConfig(
        name="small-zipf-cap1.25", T=1500, d=256, E=32, k=2, d_ff=384, capacity_factor=1.25,
        gate_bias="zipf", zipf_s=1.2, zipf_c=ZIPF_C_E64),
    "small-hybrid-top8": LayerConfig(
        name="small-hybrid-top8", T=777, d=128, E=16, k=8, d_ff=320, capacity_factor=None,
        temperature=0.2),
    "small-clusters-cap1.0": LayerConfig(
        name="small-clusters-cap1.0", T=2048, d=128, E=64, k=2, d_ff=256, capacity_factor=1.0,
        x_dist="clusters", n_clusters=16, cluster_noise=0.1),
    "small-heavy-drop": LayerConfig(
        name="small-heavy-drop", T=600, d=192, E=8, k=2, d_ff=256, capacity_factor=0.25),
    "small-fp32-bwd": LayerConfig(
        name="small-fp32-bwd", T=300, d=96, E=8, k=2, d_ff=160, capacity_factor=1.0,
        dtype="f32"),
    # average bucket >= 1024 rows: 256-row buckets and GEMM tiles on CTA pairs
    "small-pair-tiles": LayerConfig(
        name="small-pair-tiles", T=2500, d=256, E=4, k=2, d_ff=384, capacity_factor=1.0),
    # pair tiles with buckets of an odd and an even number of 128-row tiles (the odd ones end in
    # a 128-row tile), and output widths past one 256-column tile with ragged last tiles
    "small-pair-odd": LayerConfig(
        name="small-pair-odd", T=2300, d=320, E=4, k=2, d_ff=448, capacity_factor=None),
    "small-max-e256-k8": LayerConfig(
        name="small-max-e256-k8", T=513, d=128, E=256, k=8, d_ff=128, capacity_factor=None,
        temperature=0.5),
    # fp32 with row lengths that are no multiple of a 16-byte vector
    "small-fp32-ragged": LayerConfig(
        name="small-fp32-ragged", T=123, d=37, E=5, k=3, d_ff=45, capacity_factor=1.5,
        dtype="f32"),
    # dense soft routing (k = E): every expert on every token
    "small-dense-e8": LayerConfig(
        name="small-dense-e8", T=300, d=128, E=8, k=8, d_ff=192, capacity_factor=None,
        temperature=0.2),
    "small-dense-e12-cap0.5": LayerConfig(
        name="small-dense-e12-cap0.5", T=700, d=128, E=12, k=12, d_ff=128, capacity_factor=0.5,
        gate_bias="zipf", zipf_s=1.2, zipf_c=ZIPF_C_E64),
    "small-dense-e16-pairs": LayerConfig(
        name="small-dense-e16-pairs", T=1100, d=128, E=16, k=16, d_ff=128, capacity_factor=None,
        temperature=0.5),
    # dense routing past 32 experts: the gate-weight gradient dz^T x (and the soft balance
    # loss's dz Wg) run on the tensor cores from the dense dz rows
    "small-dense-e40": LayerConfig(
        name="small-dense-e40", T=700, d=128, E=40, k=40, d_ff=128, capacity_factor=None,
        temperature=0.5),
    "small-dense-fp32": LayerConfig(
        name="small-dense-fp32", T=100, d=40, E=10, k=10, d_ff=24, capacity_factor=None,
        temperature=0.7, dtype="f32"),
}


def get(name: str) -> LayerConfig:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name in SMALL_CASES:
        return SMALL_CASES[name]
    raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS) + sorted(SMALL_CASES)}")
