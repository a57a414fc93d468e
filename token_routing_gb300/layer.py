"""Thin torch-facing binding of the MoE layer C ABI.

PyTorch provides device memory and the stream; every step of the layer runs in the CUDA
kernels of libmoe.so. The functions carry the C names (route, dispatch, expert_ffn,
combine, backward) and only marshal pointers.
"""
import ctypes

import torch

from . import _lib as L

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}
MOE_DTYPE = {"bf16": L.MOE_BF16, "f32": L.MOE_F32}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream=None):
    st = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(st.cuda_stream)


def make_config(T, d, E, k, d_ff, capacity_factor=None, temperature=1.0, aux_loss_weight=0.01,
                has_gate_bias=False, dtype="bf16", noise_std=0.0, noise_seed=0):
    """Fill and validate a moe_config_t (raises MoeError on an invalid configuration)."""
    cfg = L.MoeConfig(T=T, d=d, E=E, k=k, d_ff=d_ff,
                      capacity_factor=0.0 if capacity_factor is None else float(capacity_factor),
                      temperature=float(temperature), aux_loss_weight=float(aux_loss_weight),
                      has_gate_bias=int(bool(has_gate_bias)), dtype=MOE_DTYPE[dtype],
                      noise_std=float(noise_std), noise_seed=int(noise_seed) & 0xFFFFFFFF)
    L.check("moe_config_init", L.load().moe_config_init(ctypes.byref(cfg)))
    return cfg


def config_from(layer_cfg, noise_std=0.0, noise_seed=0):
    """moe_config_t of a synth.LayerConfig-like record."""
    return make_config(layer_cfg.T, layer_cfg.d, layer_cfg.E, layer_cfg.k, layer_cfg.d_ff,
                       layer_cfg.capacity_factor, layer_cfg.temperature,
                       layer_cfg.aux_loss_weight, layer_cfg.gate_bias != "none", layer_cfg.dtype,
                       noise_std, noise_seed)


def workspace_bytes(cfg):
    return int(L.load().moe_workspace_bytes(ctypes.byref(cfg)))


def alloc_buffers(cfg, device="cuda", backward=True):
    """Every output and scratch buffer of one forward (+ backward) pass."""
    dt = torch.bfloat16 if cfg.dtype == L.MOE_BF16 else torch.float32
    T, d, E, k, f, R = cfg.T, cfg.d, cfg.E, cfg.k, cfg.d_ff, cfg.rows_capacity
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    act = dict(dtype=dt, device=device)
    b = dict(idx=torch.empty(T, k, **i32), w=torch.empty(T, k, **f32), counts=torch.empty(E, **i32),
             balance_loss=torch.empty(1, **f32), kept=torch.empty(E, **i32),
             offsets=torch.empty(E + 1, **i32), row_token=torch.empty(R, **i32),
             slot_row=torch.empty(T, k, **i32), n_dropped=torch.empty(1, **i32),
             Xp=torch.empty(R, d, **act), Gp=torch.empty(R, f, **act), H=torch.empty(R, f, **act),
             Yp=torch.empty(R, d, **act), y=torch.empty(T, d, **act),
             ws=torch.empty(max(workspace_bytes(cfg), 256), dtype=torch.uint8, device=device))
    if backward:
        b.update(dx=torch.empty(T, d, **act), dWg=torch.empty(E, d, **f32),
                 dW1=torch.empty(E, f, d, **act), db1=torch.empty(E, f, **f32),
                 dW2=torch.empty(E, d, f, **act), db2=torch.empty(E, d, **f32),
                 dbg=torch.empty(E, **f32), dw=torch.empty(T, k, **f32), loss=torch.empty(1, **f32))
    return b


def route(cfg, x, Wg, bg, b, stream=None, logits=None):
    """moe_route; `logits` (optional [T, E] fp32 tensor) receives the routing logits."""
    L.check("moe_route", L.load().moe_route(
        ctypes.byref(cfg), _p(x), _p(Wg), _p(bg), _p(b["idx"]), _p(b["w"]), _p(b["counts"]),
        _p(b["balance_loss"]), _p(logits), _p(b["ws"]), _s(stream)))


def soft_balance(cfg, logits, weight, P, loss, ws, stream=None):
    """Soft expert load P [E] and weight * mean_e (P_e - T/E)^2 into loss [1]."""
    L.check("moe_soft_balance", L.load().moe_soft_balance(
        ctypes.byref(cfg), _p(logits), ctypes.c_float(weight), _p(P), _p(loss), _p(ws), _s(stream)))


def soft_balance_backward(cfg, logits, P, weight, x, Wg, dx, dWg, dbg, ws, stream=None):
    """Adds the soft balance loss gradient into dx, dWg and (if given) dbg."""
    L.check("moe_soft_balance_backward", L.load().moe_soft_balance_backward(
        ctypes.byref(cfg), _p(logits), _p(P), ctypes.c_float(weight), _p(x), _p(Wg), _p(dx), _p(dWg),
        _p(dbg), _p(ws), _s(stream)))


def soft_balance_window(cfg, logits, weight, W, ring, state, P, Pbar, loss, ws, stream=None):
    """Soft load P [E] of this batch into the caller's ring [W, E] (slot state[0]), window
    mean Pbar [E] and weight * mean_e (Pbar_e - mean Pbar)^2 into loss [1]; advances state [2]
    (int32; zero it before the first batch)."""
    L.check("moe_soft_balance_window", L.load().moe_soft_balance_window(
        ctypes.byref(cfg), _p(logits), ctypes.c_float(weight), int(W), _p(ring), _p(state), _p(P), _p(Pbar),
        _p(loss), _p(ws), _s(stream)))


def soft_balance_window_backward(cfg, logits, Pbar, weight, state, x, Wg, dx, dWg, dbg, ws, stream=None):
    """Adds the window loss's gradient (through this batch only) into dx, dWg and (if given) dbg."""
    L.check("moe_soft_balance_window_backward", L.load().moe_soft_balance_window_backward(
        ctypes.byref(cfg), _p(logits), _p(Pbar), ctypes.c_float(weight), _p(state), _p(x), _p(Wg), _p(dx),
        _p(dWg), _p(dbg), _p(ws), _s(stream)))


def dispatch(cfg, idx, x, b, stream=None):
    L.check("moe_dispatch", L.load().moe_dispatch(
        ctypes.byref(cfg), _p(idx), _p(x), _p(b["kept"]), _p(b["offsets"]), _p(b["row_token"]),
        _p(b["slot_row"]), _p(b["n_dropped"]), _p(b["Xp"]), _p(b["ws"]), _s(stream)))


def expert_ffn(cfg, Xp, offsets, W1, b1, W2, b2, b, stream=None):
    L.check("moe_expert_ffn", L.load().moe_expert_ffn(
        ctypes.byref(cfg), _p(Xp), _p(offsets), _p(W1), _p(b1), _p(W2), _p(b2), _p(b["Gp"]),
        _p(b["H"]), _p(b["Yp"]), _p(b["ws"]), _s(stream)))


def combine(cfg, Yp, slot_row, w, y, stream=None):
    L.check("moe_combine", L.load().moe_combine(
        ctypes.byref(cfg), _p(Yp), _p(slot_row), _p(w), _p(y), _s(stream)))


def backward(cfg, dy, x, Wg, W1, W2, b, stream=None, want_dbg=True, want_dw=True, want_loss=True):
    """Backward from the forward's saved tensors in `b` (idx, w, offsets, row_token, slot_row,
    Xp, Gp, H, Yp, balance_loss); writes dx, dWg, dW1, db1, dW2, db2 (+ dbg, dw, loss)."""
    L.check("moe_backward", L.load().moe_backward(
        ctypes.byref(cfg), _p(dy), _p(x), _p(Wg), _p(b["idx"]), _p(b["w"]), _p(b["offsets"]),
        _p(b["row_token"]), _p(b["slot_row"]), _p(b["Xp"]), _p(b["Gp"]), _p(b["H"]), _p(b["Yp"]),
        _p(W1), _p(W2), _p(b["balance_loss"]), _p(b["dx"]), _p(b["dWg"]), _p(b["dW1"]),
        _p(b["db1"]), _p(b["dW2"]), _p(b["db2"]), _p(b["dbg"]) if want_dbg else None,
        _p(b["dw"]) if want_dw else None, _p(b["loss"]) if want_loss else None, _p(b["ws"]),
        _s(stream)))


def coselect(cfg, idx, H, stream=None):
    """Expert co-selection matrix H [E, E] int32 of the routing indices idx [T, k]."""
    L.check("moe_coselect", L.load().moe_coselect(ctypes.byref(cfg), _p(idx), _p(H), _s(stream)))


def forward(cfg, p, x, b, stream=None):
    """route -> dispatch -> expert_ffn -> combine; p holds Wg, bg, W1, b1, W2, b2."""
    route(cfg, x, p["Wg"], p.get("bg"), b, stream)
    dispatch(cfg, b["idx"], x, b, stream)
    expert_ffn(cfg, b["Xp"], b["offsets"], p["W1"], p["b1"], p["W2"], p["b2"], b, stream)
    combine(cfg, b["Yp"], b["slot_row"], b["w"], b["y"], stream)


def forward_backward(cfg, p, x, dy, b, stream=None):
    """One training step of the layer: the four forward calls, then the backward."""
    forward(cfg, p, x, b, stream)
    backward(cfg, dy, x, p["Wg"], p["W1"], p["W2"], b, stream)


def selftest_wait_timeout(mode, budget_cycles, timed_out, scratch, stream=None):
    """moe_selftest_wait_timeout: a bounded device wait that nothing satisfies (mode 0, the
    only mode: an mbarrier phase); read the resulting timeout with get_error()."""
    L.check("moe_selftest_wait_timeout", L.load().moe_selftest_wait_timeout(
        int(mode), int(budget_cycles), _p(timed_out), _p(scratch), _s(stream)))


class KernelTrace:
    """Device time of every kernel the library launches from this thread while the context
    is open (moe_trace_begin / moe_trace_end): `records` is a list of (kernel name, ms) in
    launch order. Launches on a stream being captured into a graph are not traced."""

    def __init__(self, max_launches=256):
        self.max_launches = int(max_launches)
        self.records = []

    def __enter__(self):
        L.check("moe_trace_begin", L.load().moe_trace_begin(self.max_launches))
        return self

    def __exit__(self, *exc):
        lib = L.load()
        n = lib.moe_trace_end()
        if exc[0] is not None:
            return False
        if n < 0:
            raise L.MoeError("moe_trace_end", n)
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        for i in range(n):
            L.check("moe_trace_record", lib.moe_trace_record(i, ctypes.byref(name), ctypes.byref(ms)))
            self.records.append((name.value.decode(), float(ms.value)))
        self.dropped = int(lib.moe_trace_dropped())
        return False


def get_error(stream=None):
    """Synchronise and report (and clear) the device error word."""
    L.check("moe_get_error", L.load().moe_get_error(_s(stream)))


def kernel_launches():
    return int(L.load().moe_kernel_launches())


class StepGraph:
    """One training step of the layer (route, dispatch, expert_ffn, combine, backward)
    captured once into a CUDA graph and replayed; removes the per-launch host cost of the
    step's ~20 kernels. The buffers in `b` and the tensors in `p`, `x`, `dy` are bound at
    capture time: refill them in place between replays. Warm the step up eagerly before
    capturing (the first calls on a device resolve driver entry points)."""

    def __init__(self, cfg, p, x, dy, b, stream=None):
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.graph = torch.cuda.CUDAGraph()
        n0 = kernel_launches()
        torch.cuda.synchronize()
        with torch.cuda.graph(self.graph, stream=self.stream):
            forward_backward(cfg, p, x, dy, b, self.stream)
        self.launches_per_step = kernel_launches() - n0

    def replay(self):
        self.graph.replay()
