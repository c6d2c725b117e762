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
SPLIT_PROFILE = os.path.join(ROOT, "profiles", "gqa_split_kernel_serving_mix.md")
KERNEL_SOURCES = [os.path.join(ROOT, "decode_step_attention_gb300", "csrc", f)
                  for f in ("gqa_decode.cu", "dec_device.cuh", "dec_launch.h")]


# ------------------------------------------------------------------ helpers ---
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


def profiled_traffic():
    """DRAM bytes per launch of the split pass from the committed ncu summary, if that
    summary was taken on the current kernel source (else None)."""
    try:
        text = open(SPLIT_PROFILE).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch_full:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """SM clock, max clock and clock-event reasons through NVML (read-only), every ~5 ms."""

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
            time.sleep(0.005)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self, t0, t1):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "timed region"
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
        qr, kc2, vc2 = O.qknorm_rope_kv_append(q, kn_, vn_, qn, kn, kc, vc, pos, cfg.theta,
                                               cfg.layout, cfg.eps)
        O.gqa_decode_attention(qr, kc2, vc2, lens[sl])
        spent += time.perf_counter() - t0
        nbytes += W.algorithmic_bytes(cfg.replace(B=1), lens[sl], 0)["step"]
        n += 1
        if spent >= budget_s:
            break
    return spent, nbytes, n


# ----------------------------------------------------------------- ours ---
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

    def step(ev_a=None, ev_b=None):
        dsa.rmsnorm_residual(d["x"], d["norm_w"], residual=resid, eps=cfg.eps, out=y)
        dsa.qknorm_rope_kv_append(q, d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["pos"],
                                  cfg.theta, cfg.layout, d["q_norm_w"], d["k_norm_w"], cfg.eps)
        if ev_a is not None:
            ev_a.record(stream)
        if args.window > 0:  # the windowed split pass is reached through the attention call
            dsa.gqa_decode_attn(q, d["k_cache"], d["v_cache"], d["lens"], max_len=max_len,
                                workspace=ws, out=out, num_parts=parts, window=args.window)
            if ev_b is not None:
                ev_b.record(stream)
            return
        dsa.gqa_decode_split(q, d["k_cache"], d["v_cache"], d["lens"], ws, max_len=max_len,
                             num_parts=parts)
        if ev_b is not None:
            ev_b.record(stream)
        dsa.split_merge(ws, d["lens"], out, Hkv, t_cap, max_len=max_len, num_parts=parts)

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
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_g0 = time.perf_counter()
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    t_g1 = time.perf_counter()
    barrier(world)
    ms_max = max_over_ranks(g0.elapsed_time(g1), world)
    time.sleep(0.02)

    # ---- end to end through the public API: the step's inputs copied from pinned host
    # memory and its results copied back, all inside the timed region. Timed two ways:
    # the host-staged step replayed from one CUDA graph (reported), and the eager
    # decode_step call with torch copies around it.
    # the step's host inputs, then residual, out and y, packed in one buffer each side so
    # the graph does one copy up (inputs + residual) and one copy down (residual, out, y)
    names_in = ["x", "q", "k_new", "v_new", "pos", "lens"]
    spec_in = [(k, tuple(inp[k].shape), inp[k].dtype) for k in names_in]
    spec_io = [("residual", tuple(resid.shape), resid.dtype), ("out", tuple(out.shape), out.dtype),
               ("y", tuple(y.shape), y.dtype)]
    n_in = dsa.packed_size(spec_in)
    n_up = n_in + dsa.packed_size(spec_io[:1])
    n_all = n_in + dsa.packed_size(spec_io)
    dbuf = torch.empty(n_all, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(n_all, dtype=torch.uint8).pin_memory()
    dv, _ = dsa.packed_views(spec_in + spec_io, dbuf)
    hv, _ = dsa.packed_views(spec_in + spec_io, hbuf)
    for k in names_in + ["residual"]:
        hv[k].copy_(inp[k])
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names_in + ["residual"])
    d2h = sum(t.numel() * t.element_size() for t in (resid, out, y))
    step_kw = dict(x=dv["x"], residual=dv["residual"], norm_w=d["norm_w"], y=dv["y"], q=dv["q"],
                   k_new=dv["k_new"], v_new=dv["v_new"], k_cache=d["k_cache"],
                   v_cache=d["v_cache"], pos=dv["pos"], lens=dv["lens"], out=dv["out"],
                   workspace=ws, theta=cfg.theta, layout=cfg.layout, q_norm_w=d["q_norm_w"],
                   k_norm_w=d["k_norm_w"], eps=cfg.eps, max_len=max_len, num_parts=parts,
                   window=args.window)

    def e2e_eager():
        dbuf[:n_up].copy_(hbuf[:n_up], non_blocking=True)
        dsa.decode_step(**step_kw)
        hbuf[n_in:].copy_(dbuf[n_in:], non_blocking=True)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world)

    e2e_eager_ms = timed(e2e_eager)
    e2e_graph = dsa.StepGraph(copies_in=[(hbuf[:n_up], dbuf[:n_up])],
                              copies_out=[(dbuf[n_in:], hbuf[n_in:])], **step_kw)
    e2e_ms = timed(e2e_graph.replay)
    sampler.stop()
    errs = dsa.device_errors(ws)

    if rank != 0:
        return None
    step_s = ms_max / 1e3 / args.steps
    value = whole_job_gbs(nbytes["step"], step_s, world)
    split_s = statistics.mean(split_ms) / 1e3
    peak, peak_kind = measured_hbm_peak()
    achieved = nbytes["attn_split"] / split_s / 1e9
    traffic = profiled_traffic()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        secs, cb, n = oracle_sample(cfg, inp, args.cpu_seconds)
        cpu = {"value": round(cb / secs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} of {cfg.B} sequences of the workload through the fp64 "
                         f"oracle step (K1+K2+attention), {secs:.1f} s, {cb / 1e6:.1f} MB "
                         f"algorithmic bytes"}
    clocks = sampler.summary(t_g0, t_g1)
    clocks_eager = sampler.summary(h0, h1)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 5),
        "us_per_step": round(step_s * 1e6, 2),
        "timing": "step captured once into a CUDA graph and replayed K times; "
                  "eager_us_per_step: the same four C-ABI calls issued one by one",
        "eager_us_per_step": round(eager_ms * 1e3 / args.steps, 2),
        "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                        "nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name + (f"_window{args.window}" if args.window else ""),
                   "window": args.window or None, "B": B, "hidden": cfg.hidden, "Hq": Hq, "Hkv": Hkv,
                   "D": D, "rope": cfg.layout, "theta": cfg.theta, "qk_norm": cfg.qk_norm,
                   "sum_lens": int(lens_np.sum()), "max_len": max_len, "num_parts": parts,
                   "bytes_per_step": nbytes["step"], "kv_bytes_per_step": nbytes["kv"],
                   "l2": "inputs larger than L2 (KV stream %.2f GB per step vs 129 MB L2); no flush"
                         % (nbytes["kv"] / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "gqa_split_kernel" if args.window == 0 else
                     "gqa_split_kernel + split_merge_kernel (windowed attention call)",
                     "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": nbytes["attn_split"],
                     "avg_launch_us": round(split_s * 1e6, 2)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbs(nbytes["step"], e2e_ms / 1e3 / args.steps, world), 2),
                "unit": "GB/s", "us_per_step": round(e2e_ms * 1e3 / args.steps, 2),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "StepGraph with packed staging: one pinned-host copy in (inputs + residual), "
                       "the step, one copy out (residual, out, y), one graph replay per step",
                "eager_us_per_step": round(e2e_eager_ms * 1e3 / args.steps, 2)},
        "gpu_launches": 3 * args.steps,  # graph: fused K1+K2, split pass, merge
        "clocks": clocks,
        "clocks_eager_region": clocks_eager,
        "device_errors": errs,
    }


# ------------------------------------------------------------ reference ---
def run_reference(args):
    """The CPU oracle as it stands, on a bounded sample of the workload per step."""
    cfg = W.CONFIGS[args.workload]
    inp = W.make_inputs(cfg)
    # size one step: the first sequences worth about args.ref_step_seconds of oracle time
    secs, _, n = oracle_sample(cfg, inp, args.ref_step_seconds)
    sub = {k: (v[:n] if isinstance(v, torch.Tensor) and k not in ("norm_w", "q_norm_w", "k_norm_w")
               else v) for k, v in inp.items()}
    scfg = cfg.replace(B=n)
    times, nb = [], 0
    for i in range(args.warmup + args.steps):
        s, nb, _ = oracle_sample(scfg, sub, float("inf"))
        if i >= args.warmup:
            times.append(s)
    total = sum(times)
    value = nb * args.steps / total / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
                   "sample_sequences": n},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {n} of {cfg.B} sequences per step"},
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
    res = run_ours(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
