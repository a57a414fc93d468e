"""The benchmark's algorithmic work per step (the numerators of its roofline and HBM
fractions) against the per-unit figures written out by hand for the headline workload."""
import bench
import synth


def test_headline_algorithmic_counts():
    cfg = synth.get("top2-e16-cap1.0")            # T 8192, d 1024, E 16, k 2, d_ff 4096, bf16
    N = 16036                                       # kept assignments at capacity 1024
    w = bench.algorithmic_counts(cfg, N)
    # expert FFN forward: two GEMMs of 2 N d d_ff flops each
    assert w["ffn_fwd_flops"] == 2 * (2 * 16036 * 1024 * 4096)
    assert w["ffn_bwd_flops"] == 2 * w["ffn_fwd_flops"]
    # permute: read x once (T d bf16), write N rows, read idx and write slot_row/row_token ints
    assert w["permute_bytes"] == 8192 * 1024 * 2 + 16036 * 1024 * 2 + 4 * (16036 + 8192 * 2)
    # router: read x and Wg, write idx (int32) and w (fp32) for T k slots
    assert w["router_bytes"] == 8192 * 1024 * 2 + 16 * 1024 * 2 + 8192 * 2 * (4 + 4)
    # combine: read N rows of Yp, write T rows of y, read slot_row and w
    assert w["combine_bytes"] == 16036 * 1024 * 2 + 8192 * 1024 * 2 + 8192 * 2 * (4 + 4)


def test_fp32_element_size_and_oracle_sample_scaling():
    cfg = synth.get("tiny-fp32-fwd")
    w = bench.algorithmic_counts(cfg, 512)
    assert w["combine_bytes"] == 512 * 64 * 4 + 256 * 64 * 4 + 256 * 2 * 8
    # the oracle's timed batch holds as many expert rows as a top-2 batch of `tokens` tokens
    dense = synth.get("dense-soft-e128-temp0.2")
    sample, npin = bench.oracle_sample_inputs(dense.with_(T=300, d=8, d_ff=8), 64)
    assert sample.T == 1 and npin["x"].shape == (1, 8)      # 64 * 2 // 128 rounds to 1 token
    top2 = synth.get("small-top2-cap1.0")
    sample, _ = bench.oracle_sample_inputs(top2, 100)
    assert sample.T == 100
