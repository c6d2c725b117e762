"""Benchmark of the decode-step attention block on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole block over one batch of synthetic inputs already in
HBM: RMSNorm+residual (K1), QK-norm+RoPE+KV append (K2), the split pass of the GQA
decode attention (K3) and its merge (K4), each a C-ABI call on one stream. The timed
value replays the step captured once into a CUDA graph; the same calls issued one
by one are timed too (``eager_us_per_step``), with CUDA events around every split
pass for the roofline figure. The
default workload is the largest configuration ("serving_mix": 256 ragged sequences,
16/4 heads, head_dim 128, 1.2 GB of KV per step), whose KV stream is far larger than
the 129 MB L2, so no flush is needed between steps.

Reported: ``value`` = algorithmic bytes of the step / device time of the step (GB/s,
all ranks), ``roofline`` for the split pass (its algorithmic bytes / its CUDA-event
duration inside the timed region, against the measured HBM copy bandwidth), ``e2e``
(the same metric through the public step call with the step's inputs copied from
pinned host memory and its results copied back, inside the timed region), the
oracle timed on the host as ``cpu_baseline``, and the SM clocks sampled through NVML
during the timed region.

``--impl reference`` times the CPU oracle (as it stands) on a bounded sample of the
same workload and prints the same line with ``"impl": "reference"``.

Several GPUs run independent replicas (the block has no exchange step): one process
per GPU under torchrun, a barrier and max-over-ranks time around the timed region.
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import hashlib
import json
import re
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode-attn block µs/step and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "serving_mix"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "decode_step_attention_gb300", "csrc", f)
                  for f in ("gqa_decode.cu", "dec_device.cuh")]


# ------------------------------------------------------------------ helpers ---
def split_profile(workload: str) -> str:
    """The committed ncu summary of the split pass on one workload (full-size launch)."""
    return os.path.join(ROOT, "profiles", f"gqa_split_kernel_{workload}.md")


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the split pass on `workload` from its committed ncu
    summary, if there is one taken on the current kernel source (else None)."""
    try:
        text = open(split_profile(workload)).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch_full:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """SM clock, max clock and clock-event reasons through NVML (read-only), every ~1 ms."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # 1 = SM
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            return

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.handle, ctypes.byref(rs))
        return time.perf_counter(), clk.value, rs.value

    def _loop(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            time.sleep(0.001)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self, t0, t1, where="timed region"):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:  # region shorter than the sampling period: nearest samples under load
            win = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            where = "nearest samples to the timed region"
        bits = 0
        for s in win:
            bits |= s[2]
        reasons = [n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(win), "window": where}


# ---------------------------------------------------------- distributed ---
# The block has no exchange step, so several GPUs run independent replicas: the
# process group only provides the barrier around the timed region and the
# max-over-ranks time. These helpers take the backend and device so the same code
# runs under NCCL on GPUs and under gloo on CPU.
def dist_setup(backend="nccl"):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, step_seconds_max: float, world: int) -> float:
    """Throughput of all replicas: every rank's bytes over the slowest rank's step time."""
    return world * bytes_per_step_per_rank / step_seconds_max / 1e9


# ------------------------------------------------------------- CPU oracle ---
def oracle_sample(cfg, inp, budget_s: float):
    """Time the oracle on the first sequences of the workload until ~budget_s of work.

    Returns (seconds, algorithmic bytes of the sample, number of sequences)."""
    from oracle import decode_ref as O
    f64 = lambda t: None if t is None else t.double().numpy()
    qn, kn = f64(inp["q_norm_w"]), f64(inp["k_norm_w"])
    nw = f64(inp["norm_w"])
    lens = inp["lens"].numpy()
    spent, nbytes, n = 0.0, 0, 0
    stages = {"rmsnorm_residual": 0.0, "qknorm_rope_kv_append": 0.0, "attention": 0.0}
    for b in range(cfg.B):
        L = int(lens[b])
        sl = slice(b, b + 1)
        x, r = f64(inp["x"][sl]), f64(inp["residual"][sl])
        q, kn_, vn_ = f64(inp["q"][sl]), f64(inp["k_new"][sl]), f64(inp["v_new"][sl])
        kc = f64(inp["k_cache"][sl, :, :L])
        vc = f64(inp["v_cache"][sl, :, :L])
        pos = inp["pos"].numpy()[sl]
        t0 = time.perf_counter()
        O.rmsnorm_residual(x, r, nw, cfg.eps)
        t1 = time.perf_counter()
        qr, kc2, vc2 = O.qknorm_rope_kv_append(q, kn_, vn_, qn, kn, kc, vc, pos, cfg.theta,
                                               cfg.layout, cfg.eps)
        t2 = time.perf_counter()
        O.gqa_decode_attention(qr, kc2, vc2, lens[sl])
        t3 = time.perf_counter()
        stages["rmsnorm_residual"] += t1 - t0
        stages["qknorm_rope_kv_append"] += t2 - t1
        stages["attention"] += t3 - t2
        spent += t3 - t0
        nbytes += W.algorithmic_bytes(cfg.replace(B=1), lens[sl], 0)["step"]
        n += 1
        if spent >= budget_s:
            break
    oracle_sample.stages = stages
    return spent, nbytes, n


# The oracle on every host core: independent (sequence, KV head) units, K1 with each
# sequence's first unit, one spawned process per core; every round starts on all of
# them together at a barrier.
def _bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> their exact float64 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _oracle_units_worker(units, shared, cfgd, rounds, barrier, results):
    from oracle import decode_ref as O
    eps = cfgd["eps"]
    nw = _bits_to_f64(shared["norm_w"])
    qn = None if shared["q_norm_w"] is None else _bits_to_f64(shared["q_norm_w"])
    kn = None if shared["k_norm_w"] is None else _bits_to_f64(shared["k_norm_w"])
    conv = lambda a: None if a is None else _bits_to_f64(a)
    prepared = [tuple(conv(a) for a in arrs) + (L,) for arrs, L in units]  # before the clock
    for _ in range(rounds):
        barrier.wait()
        t0 = time.perf_counter()
        for x, r, q, k_new, v_new, kc, vc, L in prepared:
            if x is not None:  # the sequence's RMSNorm rides with its first KV head
                O.rmsnorm_residual(x, r, nw, eps)
            qr, kc2, vc2 = O.qknorm_rope_kv_append(q, k_new, v_new, qn, kn, kc, vc,
                                                   np.array([L - 1]), cfgd["theta"],
                                                   cfgd["layout"], eps)
            O.gqa_decode_attention(qr, kc2, vc2, np.array([L]))
        results.put((t0, time.perf_counter()))


class OraclePool:
    """The fp64 oracle step over the first sequences of a workload (about ``max_bytes``
    algorithmic bytes) on every host core, for ``rounds`` timed rounds."""

    def __init__(self, cfg, inp, max_bytes: float, rounds: int):
        import multiprocessing as mp
        lens = inp["lens"].numpy()
        n, nbytes = 0, 0
        while n < cfg.B and nbytes < max_bytes:
            nbytes += W.algorithmic_bytes(cfg.replace(B=1), lens[n:n + 1], 0)["step"]
            n += 1
        self.sequences, self.bytes, self.rounds_left = n, nbytes, rounds
        units = [(b, g, int(lens[b])) for b in range(n) for g in range(cfg.Hkv)]
        self.procs = max(1, min(len(os.sched_getaffinity(0)), len(units)))
        share = [[] for _ in range(self.procs)]
        load = [0] * self.procs
        for u in sorted(units, key=lambda u: -u[2]):  # longest first, onto the least loaded
            i = load.index(min(load))
            share[i].append(u)
            load[i] += u[2] + 1
        bits = lambda t: (None if t is None else
                          t.contiguous().view(torch.int16).numpy().view(np.uint16))
        shared = {k: bits(inp[k]) for k in ("norm_w", "q_norm_w", "k_norm_w")}
        cfgd = {"eps": cfg.eps, "theta": cfg.theta, "layout": cfg.layout}
        G = cfg.G
        ctx = mp.get_context("spawn")
        self.barrier = ctx.Barrier(self.procs + 1, timeout=600)
        self.results = ctx.Queue()
        self.workers = []
        for part in share:
            payload = []
            for b, g, L in part:  # only this unit's rows travel to the worker
                hs, gs, bs = slice(g * G, (g + 1) * G), slice(g, g + 1), slice(b, b + 1)
                first = g == 0
                payload.append(((bits(inp["x"][bs]) if first else None,
                                 bits(inp["residual"][bs]) if first else None,
                                 bits(inp["q"][bs, hs]), bits(inp["k_new"][bs, gs]),
                                 bits(inp["v_new"][bs, gs]), bits(inp["k_cache"][bs, gs, :L]),
                                 bits(inp["v_cache"][bs, gs, :L])), L))
            p = ctx.Process(target=_oracle_units_worker,
                            args=(payload, shared, cfgd, rounds, self.barrier, self.results),
                            daemon=True)
            p.start()
            self.workers.append(p)

    def run(self) -> float:
        """One round; wall seconds from the first worker's start to the last one's end."""
        self.barrier.wait()
        spans = [self.results.get(timeout=600) for _ in self.workers]
        self.rounds_left -= 1
        return max(t1 for _, t1 in spans) - min(t0 for t0, _ in spans)

    def close(self):
        for p in self.workers:
            if self.rounds_left > 0:
                p.kill()
            p.join(timeout=60)


def oracle_all_cores(cfg, inp, max_bytes: float):
    """One timed round of the oracle on every host core; (seconds, bytes, sequences,
    processes), or None when a worker failed."""
    pool = None
    try:
        pool = OraclePool(cfg, inp, max_bytes, 1)
        secs = pool.run()
    except Exception:
        if pool is not None:
            pool.rounds_left = 1
            pool.close()
        return None
    pool.close()
    return secs, pool.bytes, pool.sequences, pool.procs


# ----------------------------------------------------------------- ours ---
EXTRA_WORKLOADS = ("llama3_8b_batched", "long_context_131k")


def workload_block(dsa, name, dev, steps, warmup, sampler):
    """The device-resident step of another workload, measured as the headline one: the
    captured step replayed ``steps`` times (events around the replays; L2 flushed before
    each step when the inputs fit in L2), its dominant kernel timed as a CUDA graph of 10
    back-to-back launches, its roofline against the measured HBM peak, the DRAM traffic of
    its committed ncu summary and the clocks sampled meanwhile."""
    cfg = W.CONFIGS[name]
    inp = W.make_inputs(cfg)
    lens_np = inp["lens"].numpy()
    max_len = int(lens_np.max())
    B, Hq, Hkv, D = cfg.B, cfg.Hq, cfg.Hkv, cfg.D
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    parts = dsa.default_parts(B, Hkv, D, max_len)
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, max_len, parts, device=dev)
    y, out = torch.empty_like(d["x"]), torch.empty_like(d["q"])
    nbytes = W.algorithmic_bytes(cfg, lens_np, parts)
    stream = torch.cuda.current_stream(dev)
    path = dsa.decode_step_path(B, Hq, Hkv, D, max_len)
    launches = dsa.decode_step_launches(B, Hq, Hkv, D, max_len)
    rope = dict(theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                k_norm_w=d["k_norm_w"], eps=cfg.eps)

    def one_kernel():
        """The roofline's launch: the whole step when it is one kernel, else the attention
        call (split pass and merge)."""
        if launches == 1:
            dsa.decode_step(d["x"], d["residual"], d["norm_w"], y, d["q"], d["k_new"],
                            d["v_new"], d["k_cache"], d["v_cache"], d["pos"], d["lens"], out, ws,
                            max_len=max_len, num_parts=parts, **rope)
        else:
            dsa.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["lens"], max_len=max_len,
                                workspace=ws, out=out, num_parts=parts)

    graph = dsa.StepGraph(x=d["x"], residual=d["residual"], norm_w=d["norm_w"], y=y, q=d["q"],
                          k_new=d["k_new"], v_new=d["v_new"], k_cache=d["k_cache"],
                          v_cache=d["v_cache"], pos=d["pos"], lens=d["lens"], out=out,
                          workspace=ws, max_len=max_len, num_parts=parts, **rope)
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
             if nbytes["kv"] < 2 * L2_BYTES else None)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pairs = []
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if flush is None:
        a0.record(stream)
        for _ in range(steps):
            graph.replay()
        b0.record(stream)
    else:
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            pairs.append((a, b))
    torch.cuda.synchronize()
    step_ms = (sum(a.elapsed_time(b) for a, b in pairs) if pairs else a0.elapsed_time(b0)) / steps
    # the kernel: a graph of 10 back-to-back launches, per launch
    g10 = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g10):
            for _ in range(10):
                one_kernel()
    stream.wait_stream(side)
    for _ in range(3):
        g10.replay()
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, steps // 10)
    k0.record(stream)
    for _ in range(reps):
        g10.replay()
    k1.record(stream)
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    kernel_us = k0.elapsed_time(k1) * 1e3 / (10 * reps)
    peak, peak_kind = measured_hbm_peak()
    kbytes = nbytes["step"] if launches == 1 else nbytes["attn"]
    achieved = kbytes / (kernel_us / 1e6) / 1e9
    return {
        "us_per_step": round(step_ms * 1e3, 2),
        "value": round(nbytes["step"] / (step_ms / 1e3) / 1e9, 2), "unit": "GB/s",
        "timing": "step captured into a CUDA graph, replayed %d times%s" % (
            steps, "" if flush is None else ", L2 flushed before each"),
        "launches_per_step": launches,
        "config": {"B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "sum_lens": int(lens_np.sum()),
                   "max_len": max_len, "num_parts": parts, "bytes_per_step": nbytes["step"]},
        "roofline": {"kernel": "gqa_split_kernel<fused> (split pass and merge in one launch)"
                     if path == dsa.STEP_STREAM else "decode_small_kernel (the whole step)"
                     if path == dsa.STEP_SHORT else "gqa_split_kernel + split_merge_kernel",
                     "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(name) if path == dsa.STEP_STREAM else None,
                     "algorithmic_bytes_per_launch": kbytes,
                     "avg_launch_us": round(kernel_us, 2),
                     "avg_launch_how": "a CUDA graph of 10 back-to-back launches, per launch"},
        "clocks": sampler.summary(t0, t2, "graph replays of this workload"),
        "device_errors": dsa.device_errors(ws),
    }


def run_ours(args, world, rank, local):
    import decode_step_attention_gb300 as dsa
    cfg = W.CONFIGS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = W.make_inputs(cfg)
    lens_np = inp["lens"].numpy()
    max_len = int(lens_np.max())
    t_cap = inp["t_cap"]
    B, Hq, Hkv, D = cfg.B, cfg.Hq, cfg.Hkv, cfg.D
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    parts = dsa.default_parts(B, Hkv, D, max_len)
    ws = dsa.alloc_workspace(B, Hq, Hkv, D, max_len, parts, device=dev)
    y = torch.empty_like(d["x"])
    out = torch.empty_like(d["q"])
    resid = d["residual"]
    q = d["q"]
    eff_lens = np.minimum(lens_np, args.window) if args.window > 0 else lens_np
    nbytes = W.algorithmic_bytes(cfg, eff_lens, parts)
    stream = torch.cuda.current_stream(dev)
    # short contexts: the whole step is one kernel; otherwise K1 + K2, then the attention
    # (split pass and merge in one cooperative launch; two launches with more CTAs than SMs)
    path = dsa.decode_step_path(B, Hq, Hkv, D, max_len, args.window)
    launches = dsa.decode_step_launches(B, Hq, Hkv, D, max_len, args.window)
    rope_kw = dict(theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                   k_norm_w=d["k_norm_w"], eps=cfg.eps)

    def step(ev_a=None, ev_b=None):
        if launches == 1:  # the one kernel, events around it (its roofline: see below)
            if ev_a is not None:
                ev_a.record(stream)
            dsa.decode_step(d["x"], resid, d["norm_w"], y, q, d["k_new"], d["v_new"],
                            d["k_cache"], d["v_cache"], d["pos"], d["lens"], out, ws,
                            max_len=max_len, num_parts=parts, window=args.window, **rope_kw)
            if ev_b is not None:
                ev_b.record(stream)
            return
        dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=resid, eps=cfg.eps, out=y)
        dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["pos"],
                                  cfg.theta, cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps)
        if ev_a is not None:
            ev_a.record(stream)
        # the split pass and its merge: one cooperative launch (two with more CTAs than SMs)
        dsa.gqa_decode_attn(q, d["k_cache"], d["v_cache"], d["lens"], max_len=max_len,
                            workspace=ws, out=out, num_parts=parts, window=args.window)
        if ev_b is not None:
            ev_b.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.05)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    start.record(stream)
    for i in range(args.steps):
        step(*evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    barrier(world)
    eager_ms = max_over_ranks(start.elapsed_time(end), world)
    split_ms = [a.elapsed_time(b) for a, b in evs]

    # ---- the same step captured once into a CUDA graph and replayed (the timed value)
    graph = dsa.StepGraph(x=d["x"], residual=resid, norm_w=d["norm_w"], y=y, q=q,
                          k_new=d["k_new"], v_new=d["v_new"], k_cache=d["k_cache"],
                          v_cache=d["v_cache"], pos=d["pos"], lens=d["lens"], out=out,
                          workspace=ws, theta=cfg.theta, layout=cfg.layout,
                          q_norm_w=d["q_norm_w"], k_norm_w=d["k_norm_w"], eps=cfg.eps,
                          max_len=max_len, num_parts=parts, window=args.window)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    # a step whose inputs fit in L2 (129 MB) is timed from a flushed L2: a 512 MB write
    # before every step, outside the events around the step
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
             if nbytes["kv"] < 2 * L2_BYTES else None)

    def timed_steps(fn):
        """Device time of args.steps calls of fn (ms), max over ranks."""
        barrier(world)
        torch.cuda.synchronize()
        if flush is None:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
        else:
            pairs = []
            for _ in range(args.steps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                pairs.append((a, b))
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in pairs)
        barrier(world)
        return max_over_ranks(ms, world)

    t_g0 = time.perf_counter()
    ms_max = timed_steps(graph.replay)
    t_g1 = time.perf_counter()

    # distribution of single steps (events around each replay, after the timed run):
    # p10 / median / p90, from a flushed L2 where the timed run flushes, else warm
    per_step = []
    for _ in range(args.steps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        per_step.append((a, b))
    torch.cuda.synchronize()
    per_step_us = sorted(a.elapsed_time(b) * 1e3 for a, b in per_step)
    step_stats = {"p10_us": round(per_step_us[len(per_step_us) // 10], 2),
                  "median_us": round(statistics.median(per_step_us), 2),
                  "p90_us": round(per_step_us[(9 * len(per_step_us)) // 10], 2)}
    hot_us = None
    if flush is not None:  # the same replays back to back with a warm L2, for comparison
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        hot_us = round(a.elapsed_time(b) * 1e3 / args.steps, 2)
    time.sleep(0.02)

    # ---- end to end through the public API, host to host: the step's inputs sit in
    # pinned host memory and its results go back there, every step inside the timed
    # region. The kernels reach that memory themselves (mapped, zero-copy), so no copy
    # step sits between them: K2 reads q, k_new, v_new and pos across the host link and
    # writes the rotated q to the device; the attention reads lens from the host and
    # writes out there; K1, on a second stream forked after K2, reads x and residual
    # from the host and writes y and the new residual back while the split pass runs.
    # Timed as one CUDA graph replay per step (reported) and eagerly; for comparison,
    # the fused step with one packed copy up and one down on a single stream.
    names_in = ["x", "residual", "q", "k_new", "v_new", "pos", "lens"]
    hin = {k: inp[k].clone().pin_memory() for k in names_in}
    hy = torch.empty(tuple(y.shape), dtype=y.dtype, pin_memory=True)
    hout = torch.empty(tuple(out.shape), dtype=out.dtype, pin_memory=True)
    q_dev = torch.empty_like(q)
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names_in)
    d2h = sum(t.numel() * t.element_size() for t in (resid, out, y))

    def k2_host():
        dsa.qknorm_rope_kv_append(hin["q"], hin["k_new"], hin["v_new"], d["k_cache"],
                                  d["v_cache"], hin["pos"], q_out=q_dev, **rope_kw)

    def attn_host():
        dsa.gqa_decode_attn(q_dev, d["k_cache"], d["v_cache"], hin["lens"], max_len=max_len,
                            workspace=ws, out=hout, num_parts=parts, window=args.window)

    def k1_host():
        dsa.rmsnorm_residual(hin["x"], d["norm_w"], residual=hin["residual"], eps=cfg.eps, out=hy)

    side = torch.cuda.Stream()

    def one_launch_host():  # short contexts: the whole step, every buffer it may, on the host
        dsa.decode_step(hin["x"], hin["residual"], d["norm_w"], hy, hin["q"], hin["k_new"],
                        hin["v_new"], d["k_cache"], d["v_cache"], hin["pos"], hin["lens"], hout,
                        ws, max_len=max_len, num_parts=parts, window=args.window, **rope_kw)

    def e2e_eager():  # the order StepGraph captures it in: K1 issued after the attention
        if path == dsa.STEP_SHORT:
            one_launch_host()
            return
        k2_host()
        fork = torch.cuda.Event()
        fork.record(stream)
        attn_host()
        side.wait_event(fork)
        with torch.cuda.stream(side):
            k1_host()
        stream.wait_stream(side)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        return timed_steps(fn)

    e2e_eager_ms = timed(e2e_eager)
    if path == dsa.STEP_SHORT:
        e2e_graph = dsa.StepGraph(step=one_launch_host)
    else:
        e2e_graph = dsa.StepGraph(prologue=k2_host, step=attn_host,
                                  branches=[dsa.GraphBranch(k1_host)])
    e2e_ms = timed(e2e_graph.replay)
    # the same step through the fused device-resident call with copy-engine staging
    spec_in = [(k, tuple(inp[k].shape), inp[k].dtype) for k in names_in]
    spec_out = [("y", tuple(y.shape), y.dtype), ("out", tuple(out.shape), out.dtype)]
    n_in = dsa.packed_size(spec_in)
    dbuf = torch.empty(n_in + dsa.packed_size(spec_out), dtype=torch.uint8, device=dev)
    hbuf = torch.empty(dbuf.numel(), dtype=torch.uint8).pin_memory()
    dv, _ = dsa.packed_views(spec_in + spec_out, dbuf)
    hv, _ = dsa.packed_views(spec_in + spec_out, hbuf)
    for k in names_in:
        hv[k].copy_(inp[k])
    r0 = dv["residual"].data_ptr() - dbuf.data_ptr()
    r1 = r0 + resid.numel() * resid.element_size()
    ce_graph = dsa.StepGraph(
        copies_in=[(hbuf[:n_in], dbuf[:n_in])],
        copies_out=[(dbuf[r0:r1], hbuf[r0:r1]), (dbuf[n_in:], hbuf[n_in:])],
        x=dv["x"], residual=dv["residual"], norm_w=d["norm_w"], y=dv["y"], q=dv["q"],
        k_new=dv["k_new"], v_new=dv["v_new"], k_cache=d["k_cache"], v_cache=d["v_cache"],
        pos=dv["pos"], lens=dv["lens"], out=dv["out"], workspace=ws, max_len=max_len,
        num_parts=parts, window=args.window, **rope_kw)
    ce_ms = timed(ce_graph.replay)
    t_e2e = time.perf_counter()
    errs = dsa.device_errors(ws)
    # the two other configurations the bandwidth bar names, measured the same way
    extra = {}
    if rank == 0 and world == 1 and args.window == 0 and cfg.name == DEFAULT_WORKLOAD \
            and not args.no_extra_workloads:
        for name in EXTRA_WORKLOADS:
            # at least 100 steps (~10 ms of replays) so the clock record holds ~10 samples
            extra[name] = workload_block(dsa, name, dev, max(args.steps, 100), args.warmup,
                                         sampler)
            torch.cuda.empty_cache()
    sampler.stop()

    if rank != 0:
        return None
    step_s = ms_max / 1e3 / args.steps
    value = whole_job_gbs(nbytes["step"], step_s, world)
    split_s = statistics.mean(split_ms) / 1e3
    split_alone_us = None
    if path == dsa.STEP_STREAM:  # for comparison: the split pass on its own (no merge)
        sa0, sa1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sa_ms = []
        for _ in range(args.steps):
            sa0.record(stream)
            dsa.gqa_decode_split(q, d["k_cache"], d["v_cache"], d["lens"], ws, max_len=max_len,
                                 num_parts=parts)
            sa1.record(stream)
            torch.cuda.synchronize()
            sa_ms.append(sa0.elapsed_time(sa1))
        split_alone_us = round(statistics.median(sa_ms) * 1e3, 2)
    if launches == 1:
        # events around one eager call also catch its host-side argument checks: time the
        # kernel instead as a CUDA graph of 10 back-to-back steps, per step
        g10 = torch.cuda.CUDAGraph()
        side10 = torch.cuda.Stream(dev)
        side10.wait_stream(stream)
        with torch.cuda.stream(side10):
            with torch.cuda.graph(g10):
                for _ in range(10):
                    step()
        stream.wait_stream(side10)
        for _ in range(3):
            g10.replay()
        torch.cuda.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(1, args.steps // 10)
        k0.record(stream)
        for _ in range(reps):
            g10.replay()
        k1.record(stream)
        torch.cuda.synchronize()
        split_s = k0.elapsed_time(k1) / 1e3 / (10 * reps)
    peak, peak_kind = measured_hbm_peak()
    kernel_bytes = nbytes["step"] if launches == 1 else nbytes["attn"]
    achieved = kernel_bytes / split_s / 1e9
    # committed captures are of full-size launches of the step's kernel without a window
    traffic = profiled_traffic(cfg.name) if path == dsa.STEP_STREAM and args.window == 0 else None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        secs, cb, n = oracle_sample(cfg, inp, args.cpu_seconds)
        stages = oracle_sample.stages
        one = {"value": round(cb / secs / 1e9, 6), "unit": "GB/s", "cores": 1,
               "sample": f"first {n} of {cfg.B} sequences of the workload through the fp64 "
                         f"oracle step (K1+K2+attention), {secs:.1f} s, {cb / 1e6:.1f} MB "
                         f"algorithmic bytes",
               "stage_seconds": {k: round(v, 4) for k, v in stages.items()}}
        # every core: about as much work as the one-core sample per core
        every = oracle_all_cores(cfg, inp, cb * len(os.sched_getaffinity(0)))
        if every is None:
            cpu = dict(one, kind="oracle")
        else:
            a_secs, a_cb, a_n, procs = every
            cpu = {"value": round(a_cb / a_secs / 1e9, 6), "unit": "GB/s", "cores": procs,
                   "kind": "oracle",
                   "sample": f"first {a_n} of {cfg.B} sequences through the fp64 oracle step, "
                             f"split into (sequence, KV head) units over {procs} processes "
                             f"started together, {a_secs:.2f} s wall, {a_cb / 1e6:.1f} MB "
                             f"algorithmic bytes",
                   "one_core": one}
    # the timed region of a short run lasts a few ms (a handful of 1 ms samples): the
    # headline record covers every replay of the step around it as well
    clocks = sampler.summary(t_g0, t_e2e, "graph replays of the step: the timed region, the "
                             "per-step and warm-L2 replays and the host-to-host replays")
    clocks_timed = sampler.summary(t_g0, t_g1)
    clocks_eager = sampler.summary(h0, h1, "eager loop")
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "us_per_step": round(step_s * 1e6, 2),
        "timing": ("step captured once into a CUDA graph and replayed K times"
                   + ("" if flush is None else ", L2 flushed before each replay, CUDA events "
                      "around each, summed")
                   + "; eager_us_per_step: the step's C-ABI calls issued one by one"),
        "eager_us_per_step": round(eager_ms * 1e3 / args.steps, 2),
        "step_us_stats": step_stats,
        "warm_l2_us_per_step": hot_us,
        "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                        "nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name + (f"_window{args.window}" if args.window else ""),
                   "window": args.window or None, "B": B, "hidden": cfg.hidden, "Hq": Hq, "Hkv": Hkv,
                   "D": D, "rope": cfg.layout, "theta": cfg.theta, "qk_norm": cfg.qk_norm,
                   "sum_lens": int(lens_np.sum()), "max_len": max_len, "num_parts": parts,
                   "bytes_per_step": nbytes["step"], "kv_bytes_per_step": nbytes["kv"],
                   "l2": ("inputs larger than L2 (KV stream %.2f GB per step vs 129 MB L2); "
                          "no flush" % (nbytes["kv"] / 1e9)) if flush is None else
                         "inputs fit in L2: a 512 MB write before every timed step (outside "
                         "the step's events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "decode_small_kernel (the whole step)" if path == dsa.STEP_SHORT
                     else "gqa_split_kernel<fused> (split pass and merge in one launch)"
                     if path == dsa.STEP_STREAM
                     else "gqa_split_kernel + split_merge_kernel (the attention call)",
                     "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_bytes,
                     "avg_launch_us": round(split_s * 1e6, 2),
                     "split_pass_alone_us": split_alone_us,
                     "avg_launch_how": ("a CUDA graph of 10 back-to-back steps, per step"
                                        if launches == 1 else
                                        "CUDA events around the attention call in the eager "
                                        "loop")},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbs(nbytes["step"], e2e_ms / 1e3 / args.steps, world), 2),
                "unit": "GB/s", "us_per_step": round(e2e_ms * 1e3 / args.steps, 2),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": ("inputs and results in pinned host memory, read and written by the one "
                        "kernel of the step itself (zero-copy); one CUDA graph replay per step"
                        if path == dsa.STEP_SHORT else
                        "inputs and results in pinned host memory, reached by the kernels "
                        "themselves (zero-copy): K2 reads q/k_new/v_new/pos from the host and "
                        "writes q to HBM (the split pass loads q with bulk copies, which take "
                        "device memory only), the attention (split pass and merge in one "
                        "launch) reads lens from the host and writes out there, K1 on a second "
                        "stream (forked after K2, issued after the attention) reads x/residual "
                        "and writes y/residual during the split pass; one CUDA graph replay "
                        "per step"),
                "eager_us_per_step": round(e2e_eager_ms * 1e3 / args.steps, 2),
                "copy_engine_us_per_step": round(ce_ms * 1e3 / args.steps, 2),
                "copy_engine_how": "the fused device call with one packed pinned-host copy "
                                   "in and copies of residual, y and out back, one stream"},
        # graph: fused K1+K2, split pass, merge; or the one-launch step
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "clocks_timed_region": clocks_timed,
        "clocks_eager_region": clocks_eager,
        "device_errors": errs,
        "workloads": extra or None,
    }


# ------------------------------------------------------- attention sublayer ---
L2_FLUSH_BYTES = 512 << 20  # written before every timed step whose inputs fit in L2
L2_BYTES = 129 << 20


def oracle_sublayer_sample(cfg, inp, wts, budget_s: float):
    """Time the oracle's attention sublayer on the first sequences until ~budget_s."""
    from oracle import decode_ref as O
    f64 = lambda t: None if t is None else t.double().numpy()
    lens = inp["lens"].numpy()
    common = dict(norm_w=f64(inp["norm_w"]), eps=cfg.eps, w_qkv=f64(wts["w_qkv"]),
                  w_o=f64(wts["w_o"]), q_norm_w=f64(inp["q_norm_w"]),
                  k_norm_w=f64(inp["k_norm_w"]), theta=cfg.theta, layout=cfg.layout, Hq=cfg.Hq,
                  Hkv=cfg.Hkv, D=cfg.D)
    spent, nbytes, n = 0.0, 0, 0
    for b in range(cfg.B):
        L = int(lens[b])
        sl = slice(b, b + 1)
        one = dict(common, x=f64(inp["x"][sl]), residual=f64(inp["residual"][sl]),
                   k_cache=f64(inp["k_cache"][sl, :, :L]), v_cache=f64(inp["v_cache"][sl, :, :L]),
                   pos=inp["pos"].numpy()[sl], lens=lens[sl])
        t0 = time.perf_counter()
        O.attention_sublayer(one)
        spent += time.perf_counter() - t0
        nbytes += W.sublayer_bytes(cfg.replace(B=1), lens[sl])["step"]
        n += 1
        if spent >= budget_s:
            break
    return spent, nbytes, n


def linear_roofline(dsa, B, N, K, dev, reps=20, seed=0):
    """Device time of one projection launch (dec_linear, y = x W^T): a CUDA graph of
    back-to-back launches over enough distinct weight copies that their total exceeds
    L2 three times, so every launch streams its weight from HBM; events around the
    replays. Returns (us per launch, algorithmic bytes, flops)."""
    wbytes = N * K * 2
    copies = int(min(64, max(2, -(-3 * (129 << 20) // wbytes))))
    g = torch.Generator(device="cpu").manual_seed(seed)
    w0 = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16).to(dev)
    ws_ = [w0] + [w0.clone() for _ in range(copies - 1)]
    x = torch.randn(B, K, generator=g).to(torch.bfloat16).to(dev)
    y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    for w in ws_:  # first calls set up per-device state outside the capture
        dsa.linear(x, w, out=y)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            for w in ws_:
                dsa.linear(x, w, out=y)
    torch.cuda.current_stream(dev).wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (reps * copies)
    # the same loop through cuBLAS (torch.nn.functional.linear), context for the roofline
    ref = torch.cuda.CUDAGraph()
    outs = [None]
    with torch.cuda.stream(side):
        torch.nn.functional.linear(x, w0)
        with torch.cuda.graph(ref):
            for w in ws_:
                outs[0] = torch.nn.functional.linear(x, w)
    torch.cuda.current_stream(dev).wait_stream(side)
    for _ in range(3):
        ref.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        ref.replay()
    b.record()
    torch.cuda.synchronize()
    us_lib = a.elapsed_time(b) * 1e3 / (reps * copies)
    nbytes = (N * K + B * K + B * N) * 2
    return us, nbytes, 2 * B * N * K, us_lib


def run_sublayer(args, world, rank, local):
    """The attention sublayer (RMSNorm, packed QKV projection, rotation + append,
    attention, output projection + residual) as the step."""
    import decode_step_attention_gb300 as dsa
    cfg = W.CONFIGS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = W.make_inputs(cfg)
    wts = W.make_projection_weights(cfg)
    lens_np = inp["lens"].numpy()
    max_len = int(lens_np.max())
    B, H, Hq, Hkv, D = cfg.B, cfg.hidden, cfg.Hq, cfg.Hkv, cfg.D
    nqkv = (Hq + 2 * Hkv) * D
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    w_qkv, w_o = wts["w_qkv"].to(dev), wts["w_o"].to(dev)
    parts = dsa.default_parts(B, Hkv, D, max_len)
    # the attention call: one launch (the short-context kernel, or the split pass and its
    # merge in one cooperative launch), two with more split CTAs than SMs
    attn_launches = 2 if dsa.decode_step_path(B, Hq, Hkv, D, max_len, args.window) == \
        dsa.STEP_THREE else 1
    eff_lens = np.minimum(lens_np, args.window) if args.window > 0 else lens_np
    nbytes = W.sublayer_bytes(cfg, eff_lens)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    resid = d["residual"]

    # ---- eager: the sublayer's kernels as separate C-ABI calls, CUDA events around each
    y = torch.empty_like(d["x"])
    qkv = torch.empty(B, nqkv, dtype=torch.bfloat16, device=dev)
    q, kn, vn = (torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev),
                 torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev),
                 torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev))
    attn = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    aws = dsa.alloc_workspace(B, Hq, Hkv, D, max_len, parts, device=dev)
    names = ["rmsnorm", "qkv_proj", "append", "attn", "o_proj"]

    def eager(evs=None):
        rec = (lambda i: evs[i].record(stream)) if evs else (lambda i: None)
        rec(0)
        dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=resid, eps=cfg.eps, out=y)
        rec(1)
        dsa.linear(y, w_qkv, out=qkv)
        rec(2)
        # the sublayer's rotation reads the packed columns in place; here they are
        # copied apart first (outside the events) so the public call can be timed
        dsa.qknorm_rope_kv_append(q, kn, vn, d["k_cache"], d["v_cache"], d["pos"], cfg.theta,
                                  cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps)
        rec(3)
        dsa.gqa_decode_attn(q, d["k_cache"], d["v_cache"], d["lens"], max_len=max_len,
                            workspace=aws, out=attn, num_parts=0, window=args.window)
        rec(4)
        dsa.linear(attn.view(B, Hq * D), w_o, resid, out=out)
        rec(5)

    for _ in range(args.warmup):
        eager()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.05)
    per = {n: [] for n in names}
    for _ in range(args.steps):
        flush.zero_()
        q.copy_(qkv[:, :Hq * D].view(B, Hq, D))
        kn.copy_(qkv[:, Hq * D:(Hq + Hkv) * D].view(B, Hkv, D))
        vn.copy_(qkv[:, (Hq + Hkv) * D:].view(B, Hkv, D))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        eager(evs)
        torch.cuda.synchronize()
        for i, n in enumerate(names):
            per[n].append(evs[i].elapsed_time(evs[i + 1]))
    per_us = {n: statistics.mean(v) * 1e3 for n, v in per.items()}
    proj = {}
    for n, (pn, pk) in (("qkv_proj", (nqkv, H)), ("o_proj", (H, Hq * D))):
        us, pb, fl, us_lib = linear_roofline(dsa, B, pn, pk, dev)
        proj[n] = {"shape_BNK": [B, pn, pk], "avg_launch_us": round(us, 3), "bytes": pb,
                   "cublas_us_same_harness": round(us_lib, 3),
                   "achieved_gbs": round(pb / (us * 1e-6) / 1e9, 1),
                   "tflops": round(fl / (us * 1e-6) / 1e12, 2),
                   "batch_tile_and_k_split": list(dsa.linear_plan(B, pn, pk))}

    # ---- the sublayer call captured into a CUDA graph (the timed value)
    ws = torch.zeros(dsa.sublayer_workspace_bytes(B, H, Hq, Hkv, D, max_len, parts),
                     dtype=torch.uint8, device=dev)
    kw = dict(x=d["x"], residual=resid, norm_w=d["norm_w"], w_qkv=w_qkv, w_o=w_o,
              k_cache=d["k_cache"], v_cache=d["v_cache"], pos=d["pos"], lens=d["lens"], out=out,
              workspace=ws, theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
              k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, num_parts=0,
              window=args.window)
    graph = dsa.StepGraph(step=dsa.attn_sublayer, **kw)

    def timed_flushed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        pairs = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            pairs.append((a, b))
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        barrier(world)
        ms = sum(a.elapsed_time(b) for a, b in pairs)
        return max_over_ranks(ms, world), t0, t1

    ms_graph, t_g0, t_g1 = timed_flushed(graph.replay)

    # ---- end to end: x, residual, pos and lens in pinned host memory and out written
    # there, read and written by the kernels themselves (zero-copy), one graph replay
    names_in = ["x", "residual", "pos", "lens"]
    hin = {k: inp[k].clone().pin_memory() for k in names_in}
    hout = torch.empty(B, H, dtype=torch.bfloat16, pin_memory=True)
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names_in)
    d2h = hout.numel() * hout.element_size() + hin["residual"].numel() * 2
    kw_e2e = dict(kw, x=hin["x"], residual=hin["residual"], pos=hin["pos"], lens=hin["lens"],
                  out=hout)
    e2e_graph = dsa.StepGraph(step=dsa.attn_sublayer, **kw_e2e)
    ms_e2e, _, _ = timed_flushed(e2e_graph.replay)
    sampler.stop()
    errs = dsa.device_errors(ws)

    if rank != 0:
        return None
    step_s = ms_graph / 1e3 / args.steps
    value = whole_job_gbs(nbytes["step"], step_s, world)
    peak, peak_kind = measured_hbm_peak()
    dom = max(per_us, key=per_us.get)
    achieved = nbytes[dom] / (per_us[dom] * 1e-6) / 1e9
    rooflines = {n: {"avg_launch_us": round(per_us[n], 2), "bytes": nbytes[n],
                     "achieved_gbs": round(nbytes[n] / (per_us[n] * 1e-6) / 1e9, 1),
                     "frac": round(nbytes[n] / (per_us[n] * 1e-6) / 1e9 / peak, 4)}
                 for n in names}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        secs, cb, n = oracle_sublayer_sample(cfg, inp, wts, args.cpu_seconds)
        cpu = {"value": round(cb / secs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} of {cfg.B} sequences through the fp64 oracle sublayer, "
                         f"{secs:.1f} s, {cb / 1e6:.1f} MB algorithmic bytes"}
    return {
        "metric": "attention sublayer (block + QKV/O projections) µs/step and achieved HBM GB/s, 1 GPU",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "us_per_step": round(step_s * 1e6, 2),
        "timing": "dec_attn_sublayer captured once into a CUDA graph; L2 flushed before every "
                  "step, CUDA events around each replay, summed",
        "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                        "nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic, random-init projection weights",
        "config": {"workload": cfg.name + "_sublayer" + (f"_window{args.window}" if args.window else ""),
                   "window": args.window or None, "B": B, "hidden": H, "Hq": Hq, "Hkv": Hkv,
                   "D": D, "sum_lens": int(lens_np.sum()), "max_len": max_len,
                   "num_parts": parts if dsa.decode_step_path(B, Hq, Hkv, D, max_len,
                                                             args.window) != dsa.STEP_SHORT
                   else None,
                   "attention_launches": attn_launches, "bytes_per_step": nbytes["step"],
                   "weight_bytes": nbytes["weights"], "kv_bytes_per_step": nbytes["kv"],
                   "l2": "flushed (512 MB write) before every timed step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "algorithmic_bytes_per_launch": nbytes[dom],
                     "avg_launch_us": round(per_us[dom], 2),
                     "timing": "eager C-ABI calls, events around each, L2 flushed per step"},
        "per_kernel_eager": rooflines,
        "projections_device": {n: dict(v, frac=round(v["achieved_gbs"] / peak, 4))
                               for n, v in proj.items()},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbs(nbytes["step"], ms_e2e / 1e3 / args.steps, world), 2),
                "unit": "GB/s", "us_per_step": round(ms_e2e * 1e3 / args.steps, 2),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "x, residual, pos and lens in pinned host memory and out (and the "
                       "new residual) written there by the sublayer's kernels themselves "
                       "(zero-copy); one CUDA graph replay per step"},
        # per step: RMSNorm, the QKV projection (head_dim 128: with the rotation as its
        # epilogue; head_dim 64: then the rotation), the attention (one launch), output
        # projection
        "gpu_launches": ((3 if D == 128 else 4) + attn_launches) * args.steps,
        "clocks": sampler.summary(t_g0, t_g1),
        "device_errors": errs,
    }


# ------------------------------------------------------------------ sampler ---
def run_sampler(args, world, rank, local):
    """The fused sampler (penalty -> temperature -> top-k -> top-p -> draw; by default the
    pages' decode_step settings) on rows of 131072 fp32 logits."""
    import decode_step_attention_gb300 as dsa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, V, L = args.rows, W.SAMPLER_VOCAB, 256
    pen, temp, top_p, top_k = args.penalty, args.temperature, args.top_p, args.top_k
    inp = W.make_sampler_inputs(B, V, args.sampler_kind, L=L, seed=0)
    z, ids, u = inp["logits"].to(dev), inp["ids"].to(dev), inp["u"].to(dev)
    out = torch.empty(B, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = B * V * 4 + B * L * 4 + B * 4 + B * 4

    def call():
        dsa.sample(z, ids, pen, temp, top_p, top_k, u=u, out=out)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.05)
    barrier(world)
    pairs = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    barrier(world)
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in pairs), world)
    # end to end: logits up from pinned host memory, the call, tokens back
    hz = inp["logits"].pin_memory()
    hout = torch.empty(B, dtype=torch.int32).pin_memory()

    def e2e():
        z.copy_(hz, non_blocking=True)
        call()
        hout.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        e2e()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    sampler.stop()
    if rank != 0:
        return None
    step_s = ms / 1e3 / args.steps
    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes / step_s / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle import sampler as S
        zz, ii, uu = inp["logits"].double().numpy(), inp["ids"].numpy(), inp["u"].double().numpy()
        spent, n = 0.0, 0
        while spent < min(args.cpu_seconds, 10.0):
            b = n % B
            c0 = time.perf_counter()
            S.sample(zz[b], ii[b], pen, temp, top_p, top_k, float(uu[b]))
            spent += time.perf_counter() - c0
            n += 1
        cpu = {"value": round(n * (V * 4 + L * 4 + 8) / spent / 1e9, 6), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{n} rows through the fp64 oracle sampler, {spent:.1f} s"}
    return {
        "metric": f"fused sampler µs per call (penalty {pen:g}, temperature {temp:g}, top-p "
                  f"{top_p:g}, top-k {top_k}) and GB/s of logits read, 1 GPU",
        "value": round(whole_job_gbs(nbytes, step_s, world), 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "us_per_step": round(step_s * 1e6, 2),
        "timing": "CUDA events around each call, L2 flushed (512 MB write) before every call",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic",
        "config": {"workload": f"sampler_{args.sampler_kind}_rows{B}_vocab{V}", "B": B, "V": V,
                   "L": L, "penalty": pen, "temperature": temp, "top_p": top_p, "top_k": top_k,
                   "l2": "flushed before every call",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "sampler_kernel", "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 5), "traffic": None,
                     "algorithmic_bytes_per_launch": nbytes,
                     "avg_launch_us": round(step_s * 1e6, 2)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbs(nbytes, ms_e2e / 1e3 / args.steps, world), 3),
                "unit": "GB/s", "us_per_step": round(ms_e2e * 1e3 / args.steps, 2),
                "h2d_bytes_per_step": B * V * 4, "d2h_bytes_per_step": B * 4},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(t0, t1),
    }


# ------------------------------------------------------------ reference ---
def run_reference(args):
    """The CPU oracle as it stands on every host core: each step is the fp64 oracle step
    over a bounded sample of the workload (its first sequences, about
    ``ref_step_seconds`` of one core's work per core), as (sequence, KV head) units on
    one spawned process per core."""
    cfg = W.CONFIGS[args.workload]
    inp = W.make_inputs(cfg)
    # size one step from the one-core rate on the first sequences
    secs, cb, _ = oracle_sample(cfg, inp, args.ref_step_seconds)
    per_core_bytes = cb / secs * args.ref_step_seconds
    pool = OraclePool(cfg, inp, per_core_bytes * len(os.sched_getaffinity(0)),
                      args.warmup + args.steps)
    try:
        times = [pool.run() for _ in range(args.warmup + args.steps)][args.warmup:]
    finally:
        pool.close()
    total = sum(times)
    value = pool.bytes * args.steps / total / 1e9
    n, procs = pool.sequences, pool.procs
    sample = (f"first {n} of {cfg.B} sequences per step through the fp64 oracle step, as "
              f"(sequence, KV head) units over {procs} processes started together")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
                   "sample_sequences": n},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": procs,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the Llama-shaped batch and the 131k context beside the default "
                         "workload")
    ap.add_argument("--sampler", action="store_true",
                    help="time the fused sampler on rows of 131072 fp32 logits")
    ap.add_argument("--rows", type=int, default=1, help="rows per sampler call")
    ap.add_argument("--sampler-kind", default="peaked", choices=["peaked", "flat", "ties", "masked"])
    ap.add_argument("--penalty", type=float, default=1.1, help="sampler: repetition penalty")
    ap.add_argument("--temperature", type=float, default=0.8,
                    help="sampler: temperature (<= 0: greedy)")
    ap.add_argument("--top-p", type=float, default=0.9, help="sampler: top-p (1: off)")
    ap.add_argument("--top-k", type=int, default=0, help="sampler: top-k (0: off)")
    ap.add_argument("--sublayer", action="store_true",
                    help="time the attention sublayer: the block plus the QKV and output "
                         "projections")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window attention over the last W tokens (0: whole sequence)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    world, rank, local = dist_setup("nccl")
    fn = run_sampler if args.sampler else run_sublayer if args.sublayer else run_ours
    res = fn(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
