"""Find the Zipf gate-bias scale c of the 64-expert skewed workload.

The "Expert Parallelism" page (section 2.1) reports a skewed load where one expert is
picked by about 40% of tokens. The skewed workload adds a fixed gate bias
bg_e = c * ln(p_e), p_e ~ (e+1)^-1.2, and this script bisects c on the seed-0 inputs so
that the share of tokens whose top-2 holds expert 0 is 0.40. The result is stored as
synth.configs.ZIPF_C_E64 (rounded to a multiple of 1/64, so it is exact in binary).

Uses only the oracle and the seeded generators:  python -m oracle.calibrate_zipf_bias
"""
import numpy as np

import synth
from oracle.moe_oracle import gate_logits, select_topk


def share_with_expert0(z0, log_p, c, k):
    idx, _ = select_topk(z0 + c * log_p[None, :], k)
    return float((idx == 0).any(axis=1).mean())


def main(target=0.40):
    cfg = synth.get("top2-e64-zipf-cap1.25").with_(zipf_c=0.0, backward=False)
    inp = synth.make_inputs(cfg)
    z0 = gate_logits(inp["x"].double().numpy(), inp["Wg"].double().numpy())
    p = np.array([(e + 1.0) ** (-cfg.zipf_s) for e in range(cfg.E)])
    log_p = np.log(p / p.sum())
    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if share_with_expert0(z0, log_p, mid, cfg.k) < target:
            lo = mid
        else:
            hi = mid
    c = round(0.5 * (lo + hi) * 64) / 64
    print(f"c = {0.5 * (lo + hi):.6f}; stored (multiple of 1/64) = {c}; "
          f"share = {share_with_expert0(z0, log_p, c, cfg.k):.4f}")
    return c


if __name__ == "__main__":
    main()
