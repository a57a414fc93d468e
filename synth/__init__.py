"""Seeded synthetic inputs and workload parameters (no arithmetic of the method)."""
from .configs import LayerConfig, WORKLOADS, SMALL_CASES, HEADLINE, get  # noqa: F401
from .generate import make_inputs, zipf_gate_bias, input_bytes  # noqa: F401
