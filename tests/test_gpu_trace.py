"""The kernel trace (moe_trace_begin / moe_trace_end / moe_trace_record) on the GPU: it names
and times every kernel a training step launches, leaves every result bit for bit as it is
without the trace, skips launches on a stream being captured, and counts the launches that
did not fit."""
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

KEYS = ("idx", "w", "offsets", "slot_row", "Xp", "H", "y", "dx", "dWg", "dW1", "db1", "dW2", "db2", "loss")


def _setup(moe, name="small-top2-cap1.0"):
    cfg = synth.get(name)
    c = moe.config_from(cfg)
    dev = P.to_dev(synth.make_inputs(cfg))
    return c, dev, moe.alloc_buffers(c, backward=True)


def test_trace_names_and_times_every_launch(moe_lib, cuda_device):
    moe = moe_lib
    c, dev, b = _setup(moe)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    plain = {k: b[k].clone() for k in KEYS}
    for k in KEYS:
        b[k].zero_()
    n0 = moe.kernel_launches()
    with moe.KernelTrace(256) as tr:
        moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    launched = moe.kernel_launches() - n0
    assert len(tr.records) == launched and tr.dropped == 0
    names = [n for n, _ in tr.records]
    for base in ("route_tc_kernel", "sort_hist_kernel", "sort_rank_kernel", "gather_kernel", "tc_gemm_kernel",
                 "combine_kernel", "combine_bwd_kernel", "router_bwd_kernel"):
        assert any(n.split("<")[0] == base for n in names), (base, names)
    assert all(ms > 0.0 for _, ms in tr.records)
    n = int(b["offsets"][-1].item())   # rows past the buckets in use are unspecified
    for k in KEYS:
        if k in ("Xp", "H"):
            assert torch.equal(b[k][:n], plain[k][:n]), k
        else:
            assert torch.equal(b[k], plain[k]), k


def test_trace_skips_captured_launches_and_counts_overflow(moe_lib, cuda_device):
    moe = moe_lib
    c, dev, b = _setup(moe)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    with moe.KernelTrace(64) as tr:
        g = moe.StepGraph(c, dev, dev["x"], dev["dy"], b)
        g.replay()
    torch.cuda.synchronize()
    assert tr.records == [] and tr.dropped == 0
    n0 = moe.kernel_launches()
    with moe.KernelTrace(3) as tr:
        moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    moe.get_error()
    assert len(tr.records) == 3
    assert tr.dropped == moe.kernel_launches() - n0 - 3
