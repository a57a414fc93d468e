"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot allocate device
memory (it takes no workspace; its scratch is a fixed array inside the library), must give
exactly what moe_dispatch gives with a caller-provided workspace.

Two calls in a row with different layer shapes check that the second call is not
disturbed by what the first left in the shared scratch array. The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu


def _noalloc_fn(lib):
    fn = lib.moe_dispatch_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 10
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_dispatch_matches_dispatch_twice(moe_lib, cuda_device):
    moe = moe_lib
    fn = _noalloc_fn(moe.load())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for name in ("small-clusters-cap1.0", "small-top2-cap1.0"):
        cfg = synth.get(name)
        inp = synth.make_inputs(cfg, with_dy=False)
        x = inp["x"].cuda()
        # routing indices from the oracle, so both entry points sort the same assignments
        npin = P.np_inputs(inp)
        idx = P.dev_i32(P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature)["idx"])
        c = moe.config_from(cfg)
        ref = moe.alloc_buffers(c, backward=False)
        moe.dispatch(c, idx, x, ref)
        out = moe.alloc_buffers(c, backward=False)
        for key in ("kept", "offsets", "row_token", "slot_row", "n_dropped", "Xp"):
            out[key].fill_(-7 if out[key].dtype == torch.int32 else 3.0)
        st = fn(ctypes.byref(c), _p(idx), _p(x), _p(out["kept"]), _p(out["offsets"]),
                _p(out["row_token"]), _p(out["slot_row"]), _p(out["n_dropped"]), _p(out["Xp"]), stream)
        assert st == 0, moe.load().moe_status_str(st)
        moe.get_error()
        n = int(ref["offsets"][-1].item())
        # integer outputs and the copied rows must match bit for bit
        for key in ("kept", "offsets", "slot_row", "n_dropped"):
            assert torch.equal(out[key], ref[key]), key
        assert torch.equal(out["row_token"][:n], ref["row_token"][:n])
        assert torch.equal(out["Xp"][:n], ref["Xp"][:n])
        assert int(out["n_dropped"].item()) == int(ref["n_dropped"].item())
        assert np.array_equal(out["kept"].cpu().numpy(), ref["kept"].cpu().numpy())


def _compare_with_dispatch(moe, fn, c, idx, x):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = moe.alloc_buffers(c, backward=False)
    moe.dispatch(c, idx, x, ref)
    out = moe.alloc_buffers(c, backward=False)
    for key in ("kept", "offsets", "row_token", "slot_row", "n_dropped", "Xp"):
        out[key].fill_(-7 if out[key].dtype == torch.int32 else 3.0)
    st = fn(ctypes.byref(c), _p(idx), _p(x), _p(out["kept"]), _p(out["offsets"]),
            _p(out["row_token"]), _p(out["slot_row"]), _p(out["n_dropped"]), _p(out["Xp"]), stream)
    assert st == 0, moe.load().moe_status_str(st)
    moe.get_error()
    n = int(ref["offsets"][-1].item())
    for key in ("kept", "offsets", "slot_row", "n_dropped"):
        assert torch.equal(out[key], ref[key]), key
    assert torch.equal(out["row_token"][:n], ref["row_token"][:n])
    assert torch.equal(out["Xp"][:n], ref["Xp"][:n])


def test_noalloc_dense_routing(moe_lib, cuda_device):
    """k = E (every expert on every token): the closed-form layout, no scratch used."""
    moe = moe_lib
    fn = _noalloc_fn(moe.load())
    cfg = synth.get("small-dense-e12-cap0.5")
    x = synth.make_inputs(cfg, with_dy=False)["x"].cuda()
    idx = torch.arange(cfg.E, dtype=torch.int32, device="cuda").repeat(cfg.T, 1).contiguous()
    _compare_with_dispatch(moe, fn, moe.config_from(cfg), idx, x)


def test_noalloc_near_the_scratch_limit(moe_lib, cuda_device):
    """A batch just under the assignment limit, with 256 experts: the sort's scratch comes
    closest to the fixed array's size here."""
    moe = moe_lib
    fn = _noalloc_fn(moe.load())
    T, E, k = 32760, 256, 8
    assert T * k <= 262144 and T * k > 262144 - 100
    rng = np.random.default_rng(5)
    idx_np = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)   # k distinct per token
    idx = torch.as_tensor(idx_np).cuda()
    x = torch.randn(T, 64, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    c = moe.make_config(T, 64, E, k, 64, capacity_factor=1.0)
    _compare_with_dispatch(moe, fn, c, idx, x)


def test_noalloc_rejects_oversized_batches(moe_lib):
    moe = moe_lib
    fn = _noalloc_fn(moe.load())
    c = moe.make_config(70000, 64, 8, 2, 64, capacity_factor=1.0)
    p = ctypes.c_void_p(256)
    assert fn(ctypes.byref(c), p, p, p, p, p, p, p, p, None) == moe.MOE_ERR_UNSUPPORTED
    c = moe.make_config(40000, 64, 16, 8, 64)
    assert fn(ctypes.byref(c), p, p, p, p, p, p, p, p, None) == moe.MOE_ERR_UNSUPPORTED
