"""Two layers stepped on two CUDA streams at once (no synchronisation between the streams):
each call's forked backward branch joins its own stream through per-call events, and the
library's shared side stream only serialises the two branches. Every output must equal, bit
for bit, the same step run alone."""
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

KEYS = ("idx", "w", "y", "dx", "dWg", "dW1", "db1", "dW2", "db2", "dw", "loss")


def _alone(moe, c, dev):
    b = moe.alloc_buffers(c, backward=True)
    moe.forward_backward(c, dev, dev["x"], dev["dy"], b)
    torch.cuda.synchronize()
    moe.get_error()
    return b


@pytest.mark.parametrize("names", [("small-top2-cap1.0", "small-clusters-cap1.0"),
                                   ("small-hybrid-top8", "small-top2-cap1.0")])
def test_concurrent_streams_match_sequential(names, moe_lib, cuda_device):
    moe = moe_lib
    runs = []
    for n in names:
        cfg = synth.get(n)
        c = moe.config_from(cfg)
        dev = P.to_dev(synth.make_inputs(cfg))
        runs.append((c, dev, _alone(moe, c, dev)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = [moe.alloc_buffers(c, backward=True) for c, _, _ in runs]
    torch.cuda.synchronize()
    for rep in range(3):
        for (c, dev, _), b, st in zip(runs, bufs, streams):
            with torch.cuda.stream(st):
                moe.forward_backward(c, dev, dev["x"], dev["dy"], b, st)
        torch.cuda.synchronize()
        moe.get_error()
        for (c, dev, ref), b in zip(runs, bufs):
            for k in KEYS:
                assert torch.equal(b[k], ref[k]), (rep, k)
