"""The C ABI library on the host: it builds, loads, exports every symbol include/moe.h
declares, and validates its arguments before touching a GPU (no compute calls here)."""
import ctypes
import math

import pytest
import torch

from oracle import moe_oracle as O


def test_exports_every_declared_symbol(moe_lib):
    lib = moe_lib.load()
    names = moe_lib.header_symbols()
    assert {"moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_backward",
            "moe_config_init", "moe_workspace_bytes", "moe_get_error", "moe_status_str"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.moe_version().decode().startswith("moe-gb300")


def test_status_strings(moe_lib):
    lib = moe_lib.load()
    for code in (0, -1, -2, -3, -4, -5):
        s = lib.moe_status_str(code).decode()
        assert s and s != "unknown status"
    assert lib.moe_status_str(7).decode() == "unknown status"


def _cfg(moe, **kw):
    base = dict(T=1000, d=256, E=8, k=2, d_ff=512, capacity_factor=1.0, temperature=1.0,
                aux_loss_weight=0.01, has_gate_bias=0, dtype=moe.MOE_BF16)
    base.update(kw)
    return moe.MoeConfig(**base)


@pytest.mark.parametrize("bad", [dict(T=-1), dict(d=0), dict(E=0), dict(E=257), dict(k=0),
                                 dict(k=9, E=16), dict(k=5, E=4), dict(d_ff=0),
                                 dict(temperature=0.0), dict(temperature=-1.0),
                                 dict(temperature=float("inf")), dict(dtype=7),
                                 dict(has_gate_bias=2), dict(capacity_factor=float("nan"))])
def test_config_init_rejects(moe_lib, bad):
    c = _cfg(moe_lib, **bad)
    assert moe_lib.load().moe_config_init(ctypes.byref(c)) == moe_lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("cf,T,k,E", [(1.0, 8192, 2, 16), (1.25, 16384, 2, 64), (1.0, 32768, 2, 256),
                                      (1.0, 1001, 2, 8), (0.25, 600, 2, 8), (1.1, 1000, 2, 8),
                                      (1.3, 777, 3, 7)])
def test_capacity_matches_oracle(moe_lib, cf, T, k, E):
    c = _cfg(moe_lib, T=T, k=k, E=E, capacity_factor=cf)
    assert moe_lib.load().moe_config_init(ctypes.byref(c)) == 0
    assert c.capacity == O.capacity(cf, T, k, E)


def test_rows_capacity_bounds_every_bucket_layout(moe_lib):
    for T, k, E, cf in [(1000, 2, 8, 1.0), (1000, 2, 8, 0.0), (5, 1, 256, 0.0), (0, 2, 8, 1.0),
                        (300, 8, 256, 0.0), (600, 2, 8, 0.25), (8192, 2, 16, 1.0), (2500, 2, 4, 1.0),
                        (16384, 8, 128, 0.0)]:
        c = _cfg(moe_lib, T=T, k=k, E=E, capacity_factor=cf)
        assert moe_lib.load().moe_config_init(ctypes.byref(c)) == 0
        C = c.capacity
        n_max = min(T * k, E * C)
        # 128-row buckets (the GEMM row tile) at every size
        assert c.row_align == 128
        # worst case: every bucket wastes row_align - 1 rows of padding
        worst = n_max + (c.row_align - 1) * min(E, n_max)
        assert c.rows_capacity >= worst and c.rows_capacity % c.row_align == 0
        if cf <= 0:
            assert C == 2 ** 31 - 1


@pytest.mark.parametrize("T,E,cf", [(16384, 128, 0.0), (700, 12, 0.5), (5, 256, 0.0), (0, 16, 0.0),
                                    (1100, 16, 0.0), (300, 8, 0.0)])
def test_dense_routing_config(moe_lib, T, E, cf):
    """k = E (dense soft routing) is accepted for any E; its bucket layout is closed-form:
    E buckets of min(T, C) rows each, padded to row_align, all within rows_capacity."""
    c = _cfg(moe_lib, T=T, k=E, E=E, capacity_factor=cf)
    assert moe_lib.load().moe_config_init(ctypes.byref(c)) == 0
    kept = min(T, c.capacity)
    B = -(-kept // c.row_align) * c.row_align
    assert E * B <= c.rows_capacity
    assert c.row_align == 128
    assert moe_lib.load().moe_workspace_bytes(ctypes.byref(c)) > 0


def test_unlimited_capacity_and_empty_batch(moe_lib):
    c = _cfg(moe_lib, T=0, capacity_factor=0.0)
    assert moe_lib.load().moe_config_init(ctypes.byref(c)) == 0
    assert c.rows_capacity == 0
    assert moe_lib.load().moe_workspace_bytes(ctypes.byref(c)) > 0


def test_workspace_grows_with_tokens(moe_lib):
    lib = moe_lib.load()
    sizes = []
    for T in (100, 1000, 10000):
        c = _cfg(moe_lib, T=T)
        assert lib.moe_config_init(ctypes.byref(c)) == 0
        sizes.append(lib.moe_workspace_bytes(ctypes.byref(c)))
    assert sizes[0] < sizes[1] < sizes[2] and all(s % 256 == 0 for s in sizes)


def test_entry_points_reject_uninitialised_config(moe_lib):
    lib = moe_lib.load()
    c = _cfg(moe_lib)  # moe_config_init not called: derived fields are 0
    p = ctypes.c_void_p(1)
    assert lib.moe_route(ctypes.byref(c), p, p, None, p, p, p, p, None, p, None) == moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_bytes(ctypes.byref(c)) == 0


def test_entry_points_reject_null_pointers(moe_lib):
    lib = moe_lib.load()
    c = _cfg(moe_lib)
    assert lib.moe_config_init(ctypes.byref(c)) == 0
    p = ctypes.c_void_p(16)
    cfg = ctypes.byref(c)
    inval = moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(cfg, None, p, None, p, p, p, p, None, p, None) == inval
    assert lib.moe_dispatch(cfg, p, p, p, p, p, p, None, p, p, None) == inval
    assert lib.moe_expert_ffn(cfg, p, p, p, p, None, p, p, p, p, p, None) == inval
    assert lib.moe_combine(cfg, p, None, p, p, None) == inval
    args = [p] * 26
    args[19] = None  # dW2
    assert lib.moe_backward(cfg, *args) == inval
    c.has_gate_bias = 1
    c2 = _cfg(moe_lib, has_gate_bias=1)
    assert lib.moe_config_init(ctypes.byref(c2)) == 0
    assert lib.moe_route(ctypes.byref(c2), p, p, None, p, p, p, p, None, p, None) == inval  # bg required


def test_entry_points_reject_misaligned_arrays(moe_lib):
    """Activation, weight and scratch arrays must start on a 16-byte boundary: a pointer one
    element into a buffer is refused before anything is launched."""
    lib = moe_lib.load()
    c = _cfg(moe_lib)
    assert lib.moe_config_init(ctypes.byref(c)) == 0
    cfg = ctypes.byref(c)
    p = ctypes.c_void_p(256)
    q = ctypes.c_void_p(256 + 2)   # one bf16 element past an aligned base
    inval = moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(cfg, q, p, None, p, p, p, p, None, p, None) == inval        # x
    assert lib.moe_dispatch(cfg, p, p, p, p, p, p, p, q, p, None) == inval           # Xp
    assert lib.moe_expert_ffn(cfg, p, p, p, q, p, p, p, p, p, p, None) == inval      # b1
    assert lib.moe_combine(cfg, p, p, p, q, None) == inval                           # y
    args = [p] * 26
    args[0] = q                                                                       # dy
    assert lib.moe_backward(cfg, *args) == inval
    assert lib.moe_dispatch_noalloc(cfg, p, q, p, p, p, p, p, p, None) == inval       # x
    # routing noise needs the workspace
    cn = _cfg(moe_lib)
    cn.noise_std = 0.1
    assert lib.moe_config_init(ctypes.byref(cn)) == 0
    assert lib.moe_route(ctypes.byref(cn), p, p, None, p, p, p, p, None, None, None) == inval


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_compute_call_without_gpu_reports_cuda_error(moe_lib):
    lib = moe_lib.load()
    c = _cfg(moe_lib, T=4, d=64, E=4, d_ff=64)
    assert lib.moe_config_init(ctypes.byref(c)) == 0
    p = ctypes.c_void_p(256)
    assert lib.moe_combine(ctypes.byref(c), p, p, p, p, None) == moe_lib.MOE_ERR_CUDA


def test_binding_make_config(moe_lib):
    c = moe_lib.make_config(1000, 256, 8, 2, 512, capacity_factor=1.25, temperature=0.2)
    assert c.capacity == math.ceil(1.25 * 1000 * 2 / 8)
    with pytest.raises(moe_lib.MoeError):
        moe_lib.make_config(10, 16, 4, 5, 16)


@pytest.mark.parametrize("kw,status", [
    (dict(), -1),                                    # fields never filled by moe_config_init
    (dict(T=1 << 30, k=4, E=8, capacity_factor=0.0), -2),   # T*k beyond 2^31 - 1
])
def test_noalloc_dispatch_gives_the_dispatch_config_errors(moe_lib, kw, status):
    """moe_dispatch_noalloc refuses a configuration with the same status as moe_dispatch,
    before touching a GPU."""
    lib = moe_lib.load()
    c = _cfg(moe_lib, **kw)
    p = ctypes.c_void_p(256)
    fn = lib.moe_dispatch_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 10
    got = fn(ctypes.byref(c), p, p, p, p, p, p, p, p, None)
    ref = lib.moe_dispatch(ctypes.byref(c), p, p, p, p, p, p, p, p, p, None)
    assert got == ref == status


def test_trace_argument_checks(moe_lib):
    """The kernel trace's host-side checks, before any CUDA call."""
    import ctypes as ct
    lib = moe_lib.load()
    assert lib.moe_trace_begin(0) == moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_trace_begin(1 << 17) == moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_trace_end() == moe_lib.MOE_ERR_INVALID_ARG        # no trace open
    name, ms = ct.c_char_p(), ct.c_float()
    assert lib.moe_trace_record(-1, ct.byref(name), ct.byref(ms)) == moe_lib.MOE_ERR_INVALID_ARG
    assert lib.moe_trace_record(1 << 20, ct.byref(name), ct.byref(ms)) == moe_lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("W,null", [(0, None), (-3, None), (4097, None), (3, "ring"), (3, "state"),
                                    (3, "Pbar")])
def test_soft_window_argument_checks(moe_lib, W, null):
    """moe_soft_balance_window refuses a bad window size or a missing buffer before any launch."""
    lib = moe_lib.load()
    c = _cfg(moe_lib)
    assert lib.moe_config_init(ctypes.byref(c)) == 0
    p = {k: ctypes.c_void_p(256) for k in ("logits", "ring", "state", "P", "Pbar", "loss", "ws")}
    if null:
        p[null] = None
    st = lib.moe_soft_balance_window(ctypes.byref(c), p["logits"], ctypes.c_float(1e-3), W, p["ring"], p["state"],
                                     p["P"], p["Pbar"], p["loss"], p["ws"], None)
    assert st == moe_lib.MOE_ERR_INVALID_ARG
    if null in ("state", "Pbar"):
        # every call here must be refused before any launch (the pointers are not real)
        st = lib.moe_soft_balance_window_backward(ctypes.byref(c), p["logits"], p["Pbar"], ctypes.c_float(1e-3),
                                                  p["state"], p["P"], p["P"], p["P"], p["P"], None, p["ws"], None)
        assert st == moe_lib.MOE_ERR_INVALID_ARG
