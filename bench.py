"""Throughput of the MoE layer (forward + backward) on GB300, through the C ABI.

One step = route -> dispatch -> expert_ffn -> combine -> backward over one batch of the
workload (default: hybrid routing, top-8 pre-selection over 128 experts then softmax(z/0.2)
over the 8, T=16384, d=1024, d_ff=4096, no capacity limit, bf16: 131,072 expert rows).
The step is captured once into a CUDA graph (the same five C-ABI calls) and replayed.
Per-call times come from one graph of eight (L2 flush, call) copies less a graph of the
flushes alone; a kernel trace (timing events around every launch) gives each kernel's own
device time, which for a kernel of a few microseconds includes its launch latency. Inputs are resident in
HBM when the timed region starts; L2 is flushed before every timed step, outside the step's
events: a 256 MB write, then a 256 MB read of another buffer that evicts the written lines
(so their write-back does not land in the step's first kernel). Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) every rank runs an independent replica on its
own batch (the layer has no exchange step on one device); value = all tokens / max time.
`--impl reference` times the fp64 CPU oracle instead, on bounded token samples.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s on 1 GB300; grouped-GEMM % BF16 peak; permute GB/s"
L2_FLUSH_BYTES = 256 << 20
STAGE_REPS = 8     # copies of (L2 flush, call) per per-call timing graph


class L2Flush:
    """Empties L2 between timed steps: writes a 256 MB buffer (twice the 129 MB L2), then reads
    another 256 MB buffer. The read evicts the written lines, so their write-back to HBM also
    happens before the next timed step instead of inside its first kernel; the step then starts
    with an L2 that holds only clean lines of an unrelated buffer."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int32, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.sink)


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, src="fallback")


REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))


def reasons_from_mask(mask):
    """Names of the active clock-event reasons in an NVML reason bit mask (nvml.h values)."""
    return [n for n, b in REASON_BITS if mask & b]


def summarise_clocks(samples):
    """samples: (sm_mhz, sm_max_mhz, reason names) tuples -> the bench line's `clocks` object."""
    if not samples:
        return None
    reasons = sorted({r for _, _, rs in samples for r in rs})
    return {"sm_mhz": statistics.median(a for a, _, _ in samples),
            "sm_max_mhz": max(b for _, b, _ in samples), "reasons": reasons, "samples": len(samples)}


class NvmlReader:
    """SM clock, maximum SM clock and clock-event reasons of one GPU, read through the NVML
    library that ships with the driver (the library nvidia-smi itself uses). Read-only."""
    NVML_CLOCK_SM = 1

    def __init__(self, uuid=None, index=0):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError("no NVML handle for the device")
        self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _clock(self, fn):
        v = self.ct.c_uint()
        if fn(self.h, self.NVML_CLOCK_SM, self.ct.byref(v)) != 0:
            raise RuntimeError("clock query failed")
        return float(v.value)

    def sm_mhz(self):
        return self._clock(self.lib.nvmlDeviceGetClockInfo)

    def sm_max_mhz(self):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def reason_mask(self):
        v = self.ct.c_ulonglong()
        if self.get_reasons(self.h, self.ct.byref(v)) != 0:
            raise RuntimeError("reason query failed")
        return int(v.value)


class PollingClockSampler:
    """Polls a reader (NvmlReader or a stand-in) every `period` seconds on a thread while the
    timed region runs, so that even a region of a few milliseconds gets several samples."""

    def __init__(self, reader, period=0.001):
        self.reader = reader
        self.period = period
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _sample(self):
        r = self.reader
        self.samples.append((r.sm_mhz(), r.sm_max_mhz(), reasons_from_mask(r.reason_mask())))

    def _run(self):
        try:
            while not self.stop_flag.is_set():
                self._sample()
                self.stop_flag.wait(self.period)
        except Exception:
            pass

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=5)
        if not self.samples:   # a region shorter than one NVML query: sample right after it
            try:
                self._sample()
            except Exception:
                pass
        out = summarise_clocks(self.samples)
        if out is not None:
            out["source"] = "nvml"
        return out


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 200 ms while running (used when the
    NVML library cannot be loaded)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        samples = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                a, b = float(f[1]), float(f[2])
            except ValueError:
                continue
            samples.append((a, b, [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]))
        out = summarise_clocks(samples)
        if out is not None:
            out["source"] = "nvidia-smi"
        return out


def make_clock_sampler(dev, local):
    """NVML polling when the library loads, else the nvidia-smi sampler."""
    try:
        import torch
        uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        uuid = f"GPU-{uuid}" if uuid is not None else None
        return PollingClockSampler(NvmlReader(uuid=uuid, index=local))
    except Exception:
        return ClockSampler(local)


GEMM_SOURCES = ["token_routing_gb300/csrc/gemm_tc_pair.cu", "token_routing_gb300/csrc/gemm_tc.cu",
                "token_routing_gb300/csrc/tc_gemm_common.cuh", "token_routing_gb300/csrc/tc_ptx.cuh",
                "token_routing_gb300/csrc/common.cuh"]


def gemm_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload):
    """DRAM bytes of one moe_expert_ffn call (its GEMM launches together) from the committed ncu
    record, if one was taken on this workload with the current GEMM sources (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_traffic.json")) as fh:
            rec = json.load(fh)
    except Exception:
        return None
    if rec.get("gemm_source_hash") != gemm_source_hash():
        return None
    w = rec.get("workloads", {}).get(workload)
    return None if w is None else w.get("expert_ffn_dram_bytes_per_call")


def algorithmic_counts(cfg, kept_rows):
    """Per-step algorithmic work: expert FLOPs and the permute / router / combine bytes
    (units: kept assignments N, tokens T)."""
    es = 2 if cfg.dtype == "bf16" else 4
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.d_ff
    N = kept_rows
    return dict(
        ffn_fwd_flops=4.0 * N * d * f,
        ffn_bwd_flops=8.0 * N * d * f,
        permute_bytes=T * d * es + N * d * es + 4.0 * (N + T * k),
        router_bytes=T * d * es + E * d * es + T * k * 8.0,
        combine_bytes=N * d * es + T * d * es + T * k * 8.0,
    )


GEMM_KINDS = {0: "ffn1", 1: "ffn2", 2: "dH", 3: "dX", 4: "wgrad", 5: "accum", 6: "wgrad_f32"}


def kernel_family(name):
    """Short label of a traced kernel name: the tcgen05 GEMMs by their epilogue kind (first
    template argument), everything else by its base name."""
    import re
    m = re.match(r"(tc_gemm_pair_kernel|tc_gemm_kernel)<(\d+)", name)
    if m:
        return GEMM_KINDS.get(int(m.group(2)), "gemm" + m.group(2))
    return name.split("<")[0]


def summarise_trace(records_per_step):
    """[[(name, ms), ...] per step] -> {family: {"launches_per_step", "us_per_launch", "us_per_step"}}."""
    steps = len(records_per_step)
    acc = {}
    for recs in records_per_step:
        for name, ms in recs:
            f = kernel_family(name)
            a = acc.setdefault(f, {"n": 0, "ms": 0.0, "names": set()})
            a["n"] += 1
            a["ms"] += ms
            a["names"].add(name)
    out = {}
    for f, a in acc.items():
        out[f] = {"launches_per_step": a["n"] / steps, "us_per_launch": a["ms"] * 1e3 / a["n"],
                  "us_per_step": a["ms"] * 1e3 / steps, "kernels": sorted(a["names"])}
    return out


def kernel_rooflines(cfg, kept, trace, peaks):
    """Algorithmic work of the path's main kernels over their own device time (from the
    kernel trace). Memory kernels against the measured HBM copy rate (bytes: reads + writes
    the operation needs once); the tcgen05 GEMMs against the measured burst bf16 rate (each
    traced kernel runs alone). Work per launch, N = kept assignments:
      route_tc_kernel     T d es + E d es + T k 8            (x, Wg in; idx, w out)
      sort + gather       T d es + N d es + 4 (N + T k)      (the permute)
      combine_kernel      N d es + T d es + T k 8
      combine_bwd_kernel  T d es + 2 N d es + T k 12         (dy, Yp, w, slot_row in; dYp, dw out)
      router_bwd_kernel   N d es + T d es + T k 12           (dXp, routing in; dx out)
      each expert GEMM    2 N d d_ff flop (Ffn1, Ffn2, dH, dX, each of the two weight gradients;
                          a row GEMM's time is that of its launches together)"""
    es = 2 if cfg.dtype == "bf16" else 4
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.d_ff
    N = kept
    mem = {
        "route": (["route_tc_kernel", "route_kernel"], T * d * es + E * d * es + T * k * 8.0),
        "dispatch": (["sort_hist_kernel", "sort_rank_kernel", "gather_kernel", "dense_layout_kernel"], T * d * es + N * d * es + 4.0 * (N + T * k)),
        "combine": (["combine_kernel"], N * d * es + T * d * es + T * k * 8.0),
        "combine_bwd": (["combine_bwd_kernel"], T * d * es + 2.0 * N * d * es + T * k * 12.0),
        "router_bwd": (["router_bwd_kernel", "router_bwd_wide_kernel"], N * d * es + T * d * es + T * k * 12.0),
    }
    out = {}
    for label, (fams, nbytes) in mem.items():
        us = sum(trace[f]["us_per_step"] for f in fams if f in trace)
        if us <= 0:
            continue
        gbs = nbytes / (us * 1e-6) / 1e9
        out[label] = {"kernels": [f for f in fams if f in trace], "us": us, "algorithmic_mb": nbytes / 1e6,
                      "gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "bound": "hbm"}
    # a row GEMM (Ffn1, Ffn2, dH, dX) is one or two launches (CTA-pair bodies + one-CTA tails):
    # its time is their sum; the weight gradients are two whole GEMMs (dW2, dW1) per step
    for fam in ("ffn1", "ffn2", "dH", "dX", "wgrad"):
        if fam not in trace:
            continue
        t = trace[fam]
        us = t["us_per_step"] / 2.0 if fam == "wgrad" else t["us_per_step"]
        flops = 2.0 * N * d * f
        tf = flops / (us * 1e-6) / 1e12
        out[fam] = {"us": us, "launches_per_step": t["launches_per_step"],
                    "tflops": tf, "frac": tf / peaks["bf16_tflops"], "bound": "tensor"}
    return out


def oracle_step(cfg, npin):
    from oracle import moe_oracle as O
    C = O.capacity(cfg.capacity_factor, cfg.T, cfg.k, cfg.E)
    fwd = O.forward(npin, cfg.k, cfg.temperature, C)
    O.backward(npin, fwd, npin["dy"])
    return fwd


def oracle_sample_inputs(cfg, tokens):
    """A batch of the workload holding as many expert rows (tokens x k) as a top-2 batch of
    `tokens` tokens, so that the oracle's time stays bounded for large k (dense routing)."""
    import synth
    sample = cfg.with_(T=max(1, min(cfg.T, tokens * 2 // cfg.k)))
    inp = synth.make_inputs(sample)
    return sample, {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def max_over_ranks(values, world, device=None):
    """Per-rank timings -> the maximum of each over all ranks (every rank gets the same list).
    One process per GPU: the job is as slow as its slowest replica."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: every replica's tokens over the slowest replica's step time."""
    return tokens_per_rank * world / (ms * 1e-3)


def cpu_baseline(cfg, tokens):
    """The fp64 oracle, as it stands, on one batch of `tokens` tokens of the same workload."""
    sample, npin = oracle_sample_inputs(cfg, tokens)
    t0 = time.perf_counter()
    oracle_step(sample, npin)
    dt = time.perf_counter() - t0
    return {"value": sample.T / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"one fwd+bwd step of a {sample.T}-token batch of {cfg.name} "
                      f"(numpy fp64, BLAS threads = host cores), {dt:.1f} s"}


def run_reference(args, cfg):
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    sample, npin = oracle_sample_inputs(cfg, args.ref_tokens)
    for _ in range(args.warmup):
        oracle_step(sample, npin)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(sample, npin)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = sample.T / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
                       "d_ff": cfg.d_ff, "capacity_factor": cfg.capacity_factor,
                       "temperature": cfg.temperature, "sample_tokens_per_step": sample.T},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{sample.T}-token batches of {cfg.name} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def batched_call_us(calls, flush, stream, steps):
    """Device time (us) of each call in `calls` (name -> fn(stream)): one CUDA graph of
    STAGE_REPS copies of (L2 flush, call) less a graph of the STAGE_REPS flushes alone, over
    STAGE_REPS. The graph's launch overhead is spread over the copies, the flush time is taken
    out, and every copy of the call starts with a flushed L2. Mean of `steps` replays after one
    unmeasured replay."""
    import torch
    dev = flush.w.device
    cap = torch.cuda.Stream(dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g, stream=cap):
            for _ in range(STAGE_REPS):
                flush.zero_()
                if fn is not None:
                    fn(cap)
        return g

    def replay_ms(g):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    graphs = {n: capture(fn) for n, fn in calls.items()}
    flush_graph = capture(None)
    out = {n: 0.0 for n in calls}
    for i in range(steps + 1):
        f_ms = replay_ms(flush_graph)
        for n, g in graphs.items():
            t_ms = replay_ms(g)
            if i >= 1:
                out[n] += max(t_ms - f_ms, 0.0) * 1e3 / STAGE_REPS / steps
    return out


def time_extras(moe, c, cfg, d_in, b, flush, stream, steps):
    """Device time (us) of the optional calls on the same workload (batched_call_us): the
    co-selection matrix, routing with training noise, and the soft balance loss forward and
    backward."""
    import torch
    dev = d_in["x"].device
    cn = moe.config_from(cfg, noise_std=0.1, noise_seed=1)
    H = torch.empty(cfg.E, cfg.E, dtype=torch.int32, device=dev)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    P = torch.empty(cfg.E, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    dx = torch.zeros_like(b["dx"])
    dWg = torch.zeros_like(b["dWg"])
    calls = {
        "route_us": lambda st: moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, st),
        "route_noisy_us": lambda st: moe.route(cn, d_in["x"], d_in["Wg"], d_in["bg"], b, st),
        "route_with_logits_us": lambda st: moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, st, logits=logits),
        "coselect_us": lambda st: moe.coselect(c, b["idx"], H, st),
        "soft_balance_us": lambda st: moe.soft_balance(c, logits, 1e-3, P, loss, b["ws"], st),
        "soft_balance_backward_us": lambda st: moe.soft_balance_backward(c, logits, P, 1e-3, d_in["x"], d_in["Wg"],
                                                                         dx, dWg, None, b["ws"], st),
    }
    out = batched_call_us(calls, flush, stream, steps)
    moe.get_error(stream)
    out["note"] = (f"per call: a CUDA graph of {STAGE_REPS} (L2 flush, call) copies minus the flushes alone; "
                   "noise_std 0.1; soft-balance weight 1e-3")
    return out


def profile_call(args, moe, c, d_in, b, flush, stream, forward_only):
    """For a profiler run: `--warmup` eager forward (+ backward) steps, then `--steps` calls of
    the one C-ABI call named by --profile, each after an L2 flush; prints no JSON line."""
    import torch

    def fwd():
        moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, stream)
        moe.dispatch(c, b["idx"], d_in["x"], b, stream)
        moe.expert_ffn(c, b["Xp"], b["offsets"], d_in["W1"], d_in["b1"], d_in["W2"], d_in["b2"], b, stream)
        moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"], stream)

    calls = {
        "route": lambda: moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, stream),
        "dispatch": lambda: moe.dispatch(c, b["idx"], d_in["x"], b, stream),
        "expert_ffn": lambda: moe.expert_ffn(c, b["Xp"], b["offsets"], d_in["W1"], d_in["b1"], d_in["W2"],
                                             d_in["b2"], b, stream),
        "combine": lambda: moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"], stream),
        "backward": lambda: moe.backward(c, d_in["dy"], d_in["x"], d_in["Wg"], d_in["W1"], d_in["W2"], b, stream),
    }
    calls["step"] = lambda: (fwd(), calls["backward"]())
    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        if not forward_only:
            calls["backward"]()
    for _ in range(args.steps):
        flush.zero_()
        calls[args.profile]()
    torch.cuda.synchronize()
    moe.get_error(stream)
    print(f"profiled {args.profile} x{args.steps} after {args.warmup} warm-up steps "
          f"({c.T} tokens, {moe.kernel_launches()} kernel launches in all)", file=sys.stderr)
    return 0


def run_ours(args, cfg):
    import torch
    import synth
    import token_routing_gb300 as moe

    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load()

    # each replica draws its own batch (seed = rank); weights are the same recipe
    inp = synth.make_inputs(cfg, seed=cfg.seed + rank)
    d_in = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    c = moe.config_from(cfg)
    forward_only = args.profile in ("route", "dispatch", "expert_ffn", "combine")
    b = moe.alloc_buffers(c, device=dev, backward=not forward_only)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    if args.profile:
        return profile_call(args, moe, c, d_in, b, flush, stream, forward_only)

    names = ["route", "dispatch", "expert_ffn", "combine", "backward"]

    def step(evs=None):
        if evs: evs[0].record(stream)
        moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, stream)
        if evs: evs[1].record(stream)
        moe.dispatch(c, b["idx"], d_in["x"], b, stream)
        if evs: evs[2].record(stream)
        moe.expert_ffn(c, b["Xp"], b["offsets"], d_in["W1"], d_in["b1"], d_in["W2"], d_in["b2"], b, stream)
        if evs: evs[3].record(stream)
        moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"], stream)
        if evs: evs[4].record(stream)
        moe.backward(c, d_in["dy"], d_in["x"], d_in["Wg"], d_in["W1"], d_in["W2"], b, stream)
        if evs: evs[5].record(stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    moe.get_error(stream)
    kept = int(b["kept"].sum().item())

    # per-call device times: STAGE_REPS copies of (L2 flush, call) captured into one CUDA graph,
    # minus a graph of the flushes alone, over STAGE_REPS: the graph's launch overhead is spread
    # over the copies and the flush time is taken out; every call starts with a flushed L2
    calls = {
        "route": lambda st: moe.route(c, d_in["x"], d_in["Wg"], d_in["bg"], b, st),
        "dispatch": lambda st: moe.dispatch(c, b["idx"], d_in["x"], b, st),
        "expert_ffn": lambda st: moe.expert_ffn(c, b["Xp"], b["offsets"], d_in["W1"], d_in["b1"], d_in["W2"],
                                                d_in["b2"], b, st),
        "combine": lambda st: moe.combine(c, b["Yp"], b["slot_row"], b["w"], b["y"], st),
        "backward": lambda st: moe.backward(c, d_in["dy"], d_in["x"], d_in["Wg"], d_in["W1"], d_in["W2"], b, st),
    }
    stage_ms = {n: us * 1e-3 for n, us in batched_call_us({n: calls[n] for n in names}, flush, stream,
                                                          args.steps).items()}
    moe.get_error(stream)
    # kernel trace: every kernel's own device time (timing events around each launch on its
    # stream), eager steps with L2 flushed before each
    trace_recs = []
    for i in range(args.steps + 1):
        flush.zero_()
        # ~1 ms of GPU spin after the flush, so that the host has queued the whole traced step
        # before its first kernel runs: no launch latency inside any kernel's event window
        torch.cuda._sleep(2_000_000)
        with moe.KernelTrace(512) as tr:
            step()
        if i >= 1:
            trace_recs.append(tr.records)
    moe.get_error(stream)
    trace = summarise_trace(trace_recs)
    # eager pass (plain calls, host launch gaps included) for reference
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    eager_ms = 0.0
    for i in range(args.steps):
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        eager_ms += e0.elapsed_time(e1) / args.steps
    moe.get_error(stream)

    # timed pass: the same step captured once into a CUDA graph and replayed
    graph = moe.StepGraph(c, d_in, d_in["x"], d_in["dy"], b)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize(dev)
    moe.get_error(stream)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = make_clock_sampler(dev, local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev0[i].record(stream)
        graph.replay()
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    moe.get_error(stream)
    if world > 1:
        torch.distributed.barrier()
    launches = graph.launches_per_step * args.steps
    ms = sum(a.elapsed_time(z) for a, z in zip(ev0, ev1)) / args.steps
    ms = max_over_ranks([ms], world, dev)[0]

    # end to end through the public API: every step copies its x and dy from pinned host memory
    # and reads its loss back to pinned host memory. Sequential: copy, step, read back, one after
    # the other. Pipelined (the reported e2e): two device input buffers, each with its own
    # captured step; the next step's inputs are copied on a copy stream while the current step
    # runs; the loss of every step is copied back without a host wait. No L2 flush between
    # steps here: the step's working set (weights, activations, workspace) exceeds the L2.
    x_h = inp["x"].pin_memory()
    dy_h = inp["dy"].pin_memory()
    loss_h = torch.empty(args.warmup + args.steps, dtype=torch.float32).pin_memory()
    seq_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        d_in["x"].copy_(x_h, non_blocking=True)
        d_in["dy"].copy_(dy_h, non_blocking=True)
        graph.replay()
        loss_h[i:i + 1].copy_(b["loss"], non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            seq_ms.append(e0.elapsed_time(e1))
    e2e_seq = sum(seq_ms) / len(seq_ms)

    x2 = torch.empty_like(d_in["x"])
    dy2 = torch.empty_like(d_in["dy"])
    graph2 = moe.StepGraph(c, d_in, x2, dy2, b)
    bufs = [(d_in["x"], d_in["dy"], graph), (x2, dy2, graph2)]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def pipelined(n):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            bufs[0][0].copy_(x_h, non_blocking=True)
            bufs[0][1].copy_(dy_h, non_blocking=True)
            copied[0].record(copy_stream)
        for i in range(n):
            xb, dyb, g = bufs[i % 2]
            stream.wait_event(copied[i % 2])
            g.replay()
            loss_h[i:i + 1].copy_(b["loss"], non_blocking=True)
            done[i % 2].record(stream)
            if i + 1 < n:
                nx, ndy, _ = bufs[(i + 1) % 2]
                with torch.cuda.stream(copy_stream):
                    if i >= 1:
                        copy_stream.wait_event(done[(i + 1) % 2])   # step i-1 has finished with it
                    nx.copy_(x_h, non_blocking=True)
                    ndy.copy_(dy_h, non_blocking=True)
                    copied[(i + 1) % 2].record(copy_stream)
        t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1) / n

    pipelined(args.warmup)
    e2e = pipelined(args.steps)
    e2e, e2e_seq = max_over_ranks([e2e, e2e_seq], world, dev)

    extras = time_extras(moe, c, cfg, d_in, b, flush, stream, args.steps) if not args.no_extras else None

    if rank == 0:
        peaks = _peaks()
        work = algorithmic_counts(cfg, kept)
        ffn_s = stage_ms["expert_ffn"] * 1e-3
        gemm_tflops = work["ffn_fwd_flops"] / ffn_s / 1e12
        # expert_ffn is timed alone (graph copies, L2 flushed before each): the burst peak
        peak_tc = peaks["bf16_tflops"]
        permute_gbs = work["permute_bytes"] / (stage_ms["dispatch"] * 1e-3) / 1e9
        hbm = {}
        for stage, key in (("route", "router_bytes"), ("dispatch", "permute_bytes"), ("combine", "combine_bytes")):
            gbs = work[key] / (stage_ms[stage] * 1e-3) / 1e9
            hbm[stage] = {"gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "algorithmic_mb": work[key] / 1e6}
        line = {
            "metric": METRIC, "value": job_tokens_per_s(cfg.T, world, ms), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
                       "d_ff": cfg.d_ff, "capacity_factor": cfg.capacity_factor,
                       "temperature": cfg.temperature, "kept_assignments": kept,
                       "l2": "flushed before every timed step, outside its events: a 256 MB write, then a "
                             "256 MB read of another buffer (evicts the written lines)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"kernel": "tcgen05 grouped GEMM, forward pair (GEMM1+GELU, GEMM2)",
                         "bound": "tensor", "achieved": gemm_tflops, "peak": peak_tc,
                         "unit": "TFLOP/s", "frac": gemm_tflops / peak_tc,
                         "peak_source": f"{peaks['src']} bf16 burst (the call is timed alone)",
                         "units": f"4 N d d_ff flop per call, N = {kept} kept assignments",
                         "call_us": stage_ms["expert_ffn"] * 1e3,
                         "kernel_us": sum(trace[f]["us_per_step"] for f in ("ffn1", "ffn2") if f in trace),
                         "traffic": measured_traffic(cfg.name)},
            "kernel_roofline": kernel_rooflines(cfg, kept, trace, peaks),
            "kernel_trace": {f: {kk: (round(v, 2) if isinstance(v, float) else v) for kk, v in t.items()}
                             for f, t in sorted(trace.items(), key=lambda kv: -kv[1]["us_per_step"])},
            "grouped_gemm_pct_bf16_peak": 100.0 * gemm_tflops / peak_tc,
            "permute_gbs": permute_gbs,
            "permute_frac_hbm": permute_gbs / peaks["hbm_gbs"],
            "hbm_stages": hbm,
            "stage_ms": stage_ms,
            "ms_per_step_eager": eager_ms,
            "timing": "CUDA-graph replay of the five C-ABI calls; stage_ms: per call, one graph of "
                      f"{STAGE_REPS} (L2 flush, call) copies minus a graph of the flushes alone, over "
                      f"{STAGE_REPS}; kernel_trace / kernel_roofline: each kernel's own device time "
                      "(timing events around every launch, eager steps, L2 flushed before each step; "
                      "a kernel's window includes its launch latency)",
            "e2e": {"value": job_tokens_per_s(cfg.T, world, e2e), "unit": "tokens/s",
                    "h2d_bytes_per_step": x_h.numel() * x_h.element_size() + dy_h.numel() * dy_h.element_size(),
                    "d2h_bytes_per_step": 4,
                    "timing": "pipelined: step i+1's x and dy copied on a copy stream during step i "
                              "(two input buffers, one captured step each); every step's loss copied "
                              "back; events around the whole timed sequence; no L2 flush (working set > L2)",
                    "sequential_tokens_per_s": job_tokens_per_s(cfg.T, world, e2e_seq)},
            "extras": extras,
            "gpu_launches": int(launches),
            "wall_s_timed": t_wall,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_tokens)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    import synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=synth.HEADLINE)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=8192, help="tokens in the oracle's timed batch (scaled by 2/k)")
    ap.add_argument("--ref-tokens", type=int, default=1024, help="tokens per oracle step (reference arm; scaled by 2/k)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip timing the optional calls")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per batch instead of the workload's (a smaller case of the same layer)")
    ap.add_argument("--profile", choices=["route", "dispatch", "expert_ffn", "combine", "backward", "step"],
                    default=None,
                    help="for a profiler: warm up, then run only this call (or the whole eager fwd+bwd "
                         "step) --steps times, each after an L2 flush (no JSON line)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    cfg = synth.get(args.workload)
    if args.tokens is not None:
        cfg = cfg.with_(T=int(args.tokens), name=f"{cfg.name}@T{int(args.tokens)}")
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
