"""Failure detection without a GPU fault: the library's bounded wait (an mbarrier phase wait,
as in the tensor-core pipelines) gives up after its cycle budget, records
MOE_ERR_DEVICE_TIMEOUT, and the kernel returns, so the context stays usable for the layer's
next call."""
import ctypes

import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_context_survives(moe_lib, cuda_device):
    moe = moe_lib
    lib = moe.load()
    moe.get_error()                                        # start from a clean error word
    timed_out = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.zeros(4, dtype=torch.int32, device="cuda")
    budget = 20_000_000                                    # ~10 ms of SM clock
    st = lib.moe_selftest_wait_timeout(0, ctypes.c_int64(budget), ctypes.c_void_p(timed_out.data_ptr()),
                                       ctypes.c_void_p(scratch.data_ptr()), None)
    assert st == 0
    with pytest.raises(moe.MoeError) as ei:
        moe.get_error()
    assert ei.value.status == moe.MOE_ERR_DEVICE_TIMEOUT
    assert timed_out.item() == 1
    # the error word was read and cleared; the layer still runs and matches the oracle
    cfg = synth.get("small-top2-cap1.0")
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    c = moe.config_from(cfg)
    fwd, _ = P.oracle_run(cfg, npin, None, align=c.row_align)
    dev = P.to_dev(inp)
    b = moe.alloc_buffers(c, backward=False)
    moe.forward(c, dev, dev["x"], b)
    moe.get_error()
    ok = P.nontie_tokens(fwd)
    assert (b["idx"].cpu().numpy()[ok] == fwd["idx"][ok]).all()


def test_selftest_rejects_bad_arguments(moe_lib, cuda_device):
    lib = moe_lib.load()
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    inval = moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(1, ctypes.c_int64(10_000), p, p, None) == inval
    assert lib.moe_selftest_wait_timeout(2, ctypes.c_int64(10_000), p, p, None) == inval
    assert lib.moe_selftest_wait_timeout(0, ctypes.c_int64(10), p, p, None) == inval
    assert lib.moe_selftest_wait_timeout(0, ctypes.c_int64(10**12), p, p, None) == inval
    assert lib.moe_selftest_wait_timeout(0, ctypes.c_int64(10_000), None, p, None) == inval
