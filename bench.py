#!/usr/bin/env python3
"""Benchmark of the fused cross-entropy hot path on GB300 (one JSON line on stdout).

Headline: fused CE forward+backward (``foak_ce_fwd_bwd``) on the Mistral-7B-shaped
loss batch -- batch 4 x seq 1024 = 4096 rows, V = 32000, bf16 logits ~N(0, 2^2),
the last token of each sequence ignored -- in tokens/s.  Inputs are synthetic
(seeded, see ``workloads``) and resident in HBM before the timed region; every
timed step runs on its own copy of the logits (262 MB, larger than the 129 MB L2),
so no step sees another's data in cache.

Also measured in the same run (the ``secondary`` list): the packed padding-free
batch, the Llama-3 vocabulary in bf16 and fp32, the separate forward and backward
entry points, and the chunked linear+CE call when the library exports it.

``--impl reference`` times the CPU oracle (float64 C, all host cores) on bounded
samples of the same workload instead.

``--gpus N`` with N > 1 starts N ranks itself (``torch.distributed.run``, one per
GPU, NCCL) unless it already runs under torchrun.  Every rank holds its own batch of
the workload (weak scaling) and each timed step is the data-parallel per-token mean:
the rank counts its valid tokens on the device, the counts are all-reduced (NCCL, on
the device), the fused kernel divides by the total, and the ranks' partial losses
are all-reduced.  Rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "CE fwd+bwd tokens/s and HBM GB/s (% of peak), V=32k/128k bf16, 1\u00d7GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
RING_BUDGET_BYTES = 64 << 30


# ----------------------------------------------------------------------------- utils

def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return {}, "fallback"


def _peak_hbm():
    d, src = _peaks()
    for k in ("hbm_gbs", "hbm_GBps", "hbm"):
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


def _peak_bf16(sustained: bool):
    d, src = _peaks()
    keys = ("bf16_tflops_sustained",) if sustained else ("bf16_tflops",)
    for k in keys + ("bf16_tflops",):
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k]), "of measured"
    return FALLBACK_BF16_TFLOPS, "of fallback"


def _source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "cross_entropy_loss_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _row_kernel(cfg):
    """The fused row kernel the library picks for this workload, and its source files:
    rows of at most one 64 KB slice are swept once, longer rows streamed twice."""
    es = 2 if cfg["dtype"] == wl.BF16 else 4
    if cfg["V"] * es <= 65536:
        aligned = "true" if cfg["V"] * es % 16 == 0 else "false"  # dense rows, 256-byte aligned base
        return f"ce_rows_kernel<{es},true,512,{aligned}>", ("ce_rows.cu", "row_common.cuh", "common.cuh")
    return f"ce_rows_long_kernel<{es},true,512,8>", ("ce_rows_long.cu", "row_common.cuh", "common.cuh")


def _traffic(profile_name, sha):
    """Per-launch DRAM bytes from a committed ncu summary, if taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(p):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha") != sha:
        return None
    try:
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only) in a thread."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, torch_device_index: int = 0):
        self.ok = False
        self.samples = []
        self.windows = []
        self._stop = threading.Event()
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            import torch

            uuid = str(torch.cuda.get_device_properties(torch_device_index).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self._reasons_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and \
                    self._reasons_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((t, int(clk.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "NVML unavailable"}
        inside = [s for s in self.samples if any(a <= s[0] <= b for a, b in self.windows)]
        use = inside if inside else self.samples
        mhz = [s[1] for s in use]
        bits = 0
        for s in use:
            bits |= s[2]
        reasons = [n for b, n in self.REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ----------------------------------------------------------------------------- workloads

def _make(name):
    if name == "mistral":
        return wl.mistral()
    if name == "packed":
        return wl.packed()
    if name == "llama3":
        return wl.llama3(dtype=wl.BF16)
    if name == "llama3_f32":
        return wl.llama3(dtype=wl.F32)
    if name == "tiny":
        return wl.tiny()
    raise ValueError(name)


WORKLOAD_DESC = {
    "mistral": "Mistral-7B loss batch: 4x1024 tokens, V=32000, bf16 logits ~N(0,2^2), last token of each "
               "sequence -100",
    "packed": "padding-free packed batch: 8192 tokens, sequence lengths U{64..1024}, V=32000, bf16 ~N(0,2^2), "
              "first token + 30-60% prompt prefix of each sequence -100",
    "llama3": "Llama-3 vocab: N=8192, V=128256, bf16 ~N(0,3^2) + 0.01% spikes U[20,30), one all-equal row, "
              "5% rows -100",
    "llama3_f32": "Llama-3 vocab: N=8192, V=128256, fp32 ~N(0,3^2) + 0.01% spikes U[20,30), one all-equal row, "
                  "5% rows -100",
    "tiny": "tiny: N=64, V=1000, fp32 ~N(0,1), 6 rows -100",
}


def _algo_bytes(cfg, fused=True):
    """Bytes the fused pass must move: valid rows read+write, ignored rows write only, labels."""
    N, V = cfg["logits"].shape[0], cfg["V"]
    es = 2 if cfg["dtype"] == wl.BF16 else 4
    n_valid = int(((cfg["labels"] >= 0) & (cfg["labels"] < V)).sum())
    if fused:
        return (2 * n_valid + (N - n_valid)) * V * es + 8 * N
    return n_valid * V * es + 8 * N + 4 * N  # forward: read valid rows, labels, write lse


def _stated_bytes(cfg):
    N, V = cfg["logits"].shape[0], cfg["V"]
    es = 2 if cfg["dtype"] == wl.BF16 else 4
    return 2 * N * V * es


# ----------------------------------------------------------------------------- ours

def _ring(torch, x_dev, count, ring_max=None):
    size = x_dev.numel() * x_dev.element_size()
    r = max(2, min(count, RING_BUDGET_BYTES // max(size, 1), ring_max or count))
    bufs = [torch.empty_like(x_dev) for _ in range(r)]
    return bufs


def _fill(bufs, x_dev):
    for b in bufs:
        b.copy_(x_dev)


def run_ours(args, rank, world, dist):
    import torch

    import cross_entropy_loss_gb300 as ce

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index) if rank == 0 and not args.profile else None

    def upload(a, dtype):
        if dtype == wl.BF16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    def barrier(use_dist=True):
        if dist is not None and use_dist:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def fused_timing(cfg, steps, warmup, record_clocks, use_dist=True, call=None, ring_max=None):
        call = call or ce.foak_ce_fwd_bwd
        x = upload(cfg["logits"], cfg["dtype"])
        y = torch.from_numpy(cfg["labels"]).to(dev)
        N = x.shape[0]
        ws = ce.workspace(N, dev)
        bufs = _ring(torch, x, steps + warmup, ring_max)
        _fill(bufs, x)
        del x
        for i in range(warmup):
            call(bufs[i % len(bufs)], y, workspace_tensor=ws)
        if warmup and len(bufs) < steps + warmup:
            _fill(bufs, upload(cfg["logits"], cfg["dtype"]))
        barrier(use_dist)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        out = None
        for i in range(steps):
            out = call(bufs[(warmup + i) % len(bufs)], y, workspace_tensor=ws)
        e1.record(stream)
        e1.synchronize()
        t1 = time.perf_counter()
        barrier(use_dist)
        if record_clocks and sampler is not None:
            sampler.mark(t0, t1)
        ms = e0.elapsed_time(e1) / steps
        loss = float(out["loss"].item())
        err = int(out["err"].item())
        reused = len(bufs) < steps + warmup
        del bufs
        torch.cuda.empty_cache()
        return ms, loss, err, reused

    def max_over_ranks(v):
        if dist is None:
            return v
        from cross_entropy_loss_gb300 import dp

        return dp.max_over_ranks(v, device=dev)

    main = _make(args.workload)
    if args.profile and args.rows > 0:
        main = dict(main, logits=main["logits"][:args.rows], labels=main["labels"][:args.rows])
    if sampler:
        sampler.start()
    if args.profile and args.path == "chunked":
        return {"metric": "chunked linear+CE (profiling run)", "chunked": chunked_timing(ce, torch, dev, stream)}
    call = None
    if dist is not None:
        # the data-parallel step: local count -> all-reduce on the device -> fused call reading the total
        from cross_entropy_loss_gb300 import dp

        cnt_buf = torch.empty(1, dtype=torch.int64, device=dev)
        V_main = main["V"]

        def call(b, y, workspace_tensor):
            return dp.fused_step(lambda yy: ce.foak_ce_count_valid(yy, V_main, out=cnt_buf),
                                 lambda xx, yy, d: ce.foak_ce_fwd_bwd_devdenom(xx, yy, d,
                                                                               workspace_tensor=workspace_tensor),
                                 b, y)
    if args.profile and args.path == "forward":
        call = lambda b, y, workspace_tensor: ce.foak_ce_forward(b, y, workspace_tensor=workspace_tensor)  # noqa: E731
    if args.profile and args.path == "backward":
        x0 = upload(main["logits"], main["dtype"])
        y0 = torch.from_numpy(main["labels"]).to(dev)
        lse0 = ce.foak_ce_forward(x0, y0)["lse"]
        dl = torch.empty_like(x0)

        def call(b, y, workspace_tensor):
            ce.foak_ce_backward(b, y, lse0, dlogits=dl)
            return {"loss": torch.zeros(1, device=dev), "err": torch.zeros(1, dtype=torch.int32, device=dev)}
    ms, loss, err, reused = fused_timing(main, args.steps, args.warmup, True, call=call)
    ms = max_over_ranks(ms)
    if sampler:
        sampler.stop()
    N = main["logits"].shape[0]
    algo = _algo_bytes(main)
    stated = _stated_bytes(main)
    peak, peak_src = _peak_hbm()
    kernel, srcs = _row_kernel(main)
    prof_name = f"ce_fused_{args.workload}.txt"
    if args.profile and args.path in ("forward", "backward"):
        # the profiling line of a separate pass: its own bytes and kernel (the secondary entries' counts)
        es = 2 if main["dtype"] == wl.BF16 else 4
        n_val = int(((main["labels"] >= 0) & (main["labels"] < main["V"])).sum())
        if args.path == "forward":
            algo = n_val * main["V"] * es + 12 * N
            kernel, srcs = f"ce_rows_warp_kernel<{es},false>", ("ce_rows_warp.cu", "row_common.cuh", "common.cuh")
        else:
            algo = (2 * n_val + (N - n_val)) * main["V"] * es + 12 * N
            kernel, srcs = f"ce_backward_kernel<{es}>", ("ce_backward.cu", "common.cuh")
        prof_name = f"ce_{args.path}_{args.workload}.txt"
    achieved = algo / (ms * 1e-3) / 1e9
    sha = _source_sha(*srcs)
    res = {
        "metric": METRIC,
        "value": world * N / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if main["dtype"] == wl.BF16 else "f32",
        "data": "synthetic (seeded SplitMix64 + Box-Muller; no dataset)",
        "config": _config(main, args.workload),
        "parallelism": (f"dp{world}: a batch per rank, per-token mean over all ranks (valid-token count "
                        "all-reduced on the device each step, partial losses all-reduced)") if world > 1
                       else "dp1",
        "l2": "inputs larger than L2: each timed step has its own 262 MB-class logits copy"
              + (" (ring reused: steps > ring)" if reused else ""),
        # the rows whose label counts (ignored rows are in `value`, not here)
        "valid_tokens_per_s": world * int(((main["labels"] >= 0) & (main["labels"] < main["V"])).sum()) / (ms * 1e-3),
        "hbm_GBps_algorithmic": achieved,
        "hbm_GBps_stated_2NVs": stated / (ms * 1e-3) / 1e9,
        "loss": loss, "err": err,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": _traffic(prof_name, sha),
                     "algorithmic_bytes_per_launch": algo, "kernel": kernel,
                     "kernel_source_sha": sha},
        # our kernels per timed step: the fused kernel (N > 1: plus the label count; NCCL's are not ours)
        "gpu_launches": args.steps * (2 if world > 1 else 1),
    }

    if args.profile:
        return res
    # end-to-end through the public API: pinned host logits -> device, fused call, loss -> host
    if rank == 0 or dist is not None:
        res["e2e"] = e2e_timing(ce, torch, dev, stream, main, max(3, min(args.steps, 20)), upload, barrier,
                                max_over_ranks, world, dist)

    if rank == 0 and not args.quick:
        res["secondary"] = secondary(ce, torch, dev, stream, upload, fused_timing, args)
    if sampler:
        res["clocks"] = sampler.summary()
    if rank == 0:
        res["cpu_baseline"] = cpu_baseline(main)
        # the metric's second vocabulary, last on the line so a tail of the output keeps it
        by = {s.get("key"): s for s in res.get("secondary", []) if s.get("key")}
        res["v128k_bf16"] = _compact(by.get("llama3"))
        res["v128k_f32"] = _compact(by.get("llama3_f32"))
        res["packed_v32k_bf16"] = _compact(by.get("packed"))
    return res


def _compact(s):
    if not s:
        return None
    return {"workload": s["workload_key"], "ms_per_step": s["ms_per_step"], "tokens_per_s": s["tokens_per_s"],
            "GBps_algorithmic": s["GBps_algorithmic"], "frac": s["frac"], "peak": s["peak"],
            "peak_source": s["peak_source"]}


def _config(cfg, name):
    """The workload, the same keys in both arms (ours and the reference's)."""
    return {"workload": WORKLOAD_DESC[name], "N": int(cfg["logits"].shape[0]), "V": int(cfg["V"]),
            "seed": int(cfg["seed"])}


def e2e_timing(ce, torch, dev, stream, cfg, steps, upload, barrier, max_over_ranks, world, dist=None):
    """The fused call on HOST buffers through the C ABI (foak_ce_fwd_bwd_host): each step
    copies that step's pinned logits and labels to the device in row chunks, sweeps
    every chunk as it lands, and reads the loss, n_valid and error word back.  With
    several ranks each step first copies the labels, counts them on the device and
    all-reduces the count, which the host call then takes as its denominator."""
    es = 2 if cfg["dtype"] == wl.BF16 else 4
    host_x = torch.from_numpy(cfg["logits"].view(np.int16) if es == 2 else cfg["logits"]).pin_memory()
    if es == 2:
        host_x = host_x.view(torch.bfloat16)
    host_y = torch.from_numpy(cfg["labels"]).pin_memory()
    x = torch.empty(host_x.shape, dtype=host_x.dtype, device=dev)
    y = torch.empty(host_y.shape, dtype=torch.int64, device=dev)
    N = host_x.shape[0]
    ws = ce.workspace(N + 64, dev)
    out = dict(loss=torch.empty(1, dtype=torch.float32).pin_memory(),
               n_valid=torch.empty(1, dtype=torch.int32).pin_memory(),
               err=torch.empty(1, dtype=torch.int32).pin_memory())

    cnt = torch.empty(1, dtype=torch.int64, device=dev)

    def step():
        denom = 0.0
        if dist is not None:
            y.copy_(host_y, non_blocking=True)
            ce.foak_ce_count_valid(y, cfg["V"], out=cnt)
            dist.all_reduce(cnt)
            denom = float(cnt.item())
        ce.foak_ce_fwd_bwd_host(host_x, host_y, x, y, denom=denom, workspace_tensor=ws, out=out, stream=stream)

    for _ in range(3):
        step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    e1.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps)
    h2d = host_x.numel() * host_x.element_size() + host_y.numel() * 8 * (2 if dist is not None else 1)
    return {"value": world * N / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 12,
            "loss": float(out["loss"].item()), "err": int(out["err"].item()),
            "path": "foak_ce_fwd_bwd_host: pinned host logits+labels -> chunked H2D overlapped with the fused "
                    "sweep of each landed chunk -> loss, n_valid, err D2H"}


def secondary(ce, torch, dev, stream, upload, fused_timing, args):
    out = []
    peak, peak_src = _peak_hbm()
    for name in ("packed", "llama3", "llama3_f32"):
        cfg = _make(name)
        # enough calls that the first one's launch after the synchronise is amortised; every
        # buffer is larger than L2, so eight of them in turn leave nothing cached between uses
        k, w = 50, 3
        ms, loss, err, reused = fused_timing(cfg, k, w, False, use_dist=False, ring_max=8)
        algo = _algo_bytes(cfg)
        gbs = algo / (ms * 1e-3) / 1e9
        out.append({"key": name, "workload_key": f"{name}: N={cfg['logits'].shape[0]} V={cfg['V']}",
                    "path": "foak_ce_fwd_bwd", "kernel": _row_kernel(cfg)[0], "workload": WORKLOAD_DESC[name],
                    "steps": k, "ms_per_step": ms,
                    "tokens_per_s": cfg["logits"].shape[0] / (ms * 1e-3),
                    "valid_tokens_per_s": int(((cfg["labels"] >= 0) & (cfg["labels"] < cfg["V"])).sum()) / (ms * 1e-3),
                    "GBps_algorithmic": gbs,
                    "GBps_stated_2NVs": _stated_bytes(cfg) / (ms * 1e-3) / 1e9, "frac": gbs / peak,
                    "peak": peak, "peak_source": peak_src, "loss": loss, "err": err,
                    "l2": "distinct logits buffers in turn (8 at most), each larger than L2"
                          + (" (reused)" if reused else "")})
        del cfg
    # separate forward and backward on the headline workload
    cfg = _make(args.workload)
    x = upload(cfg["logits"], cfg["dtype"])
    y = torch.from_numpy(cfg["labels"]).to(dev)
    N = x.shape[0]
    ws = ce.workspace(N, dev)
    k, w = 100, 3
    bufs = _ring(torch, x, k + w, 16)  # 262 MB buffers in turn: none is in L2 when it comes back
    _fill(bufs, x)
    dl = [torch.empty_like(x) for _ in range(2)]
    for i in range(w):
        f = ce.foak_ce_forward(bufs[i], y, workspace_tensor=ws)
        ce.foak_ce_backward(bufs[i], y, f["lse"], dlogits=dl[i % 2])
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev[0].record(stream)
    fs = []
    for i in range(k):
        fs.append(ce.foak_ce_forward(bufs[(w + i) % len(bufs)], y, workspace_tensor=ws))
    ev[1].record(stream)
    for i in range(k):
        ce.foak_ce_backward(bufs[(w + i) % len(bufs)], y, fs[i]["lse"], dlogits=dl[i % 2])
    ev[2].record(stream)
    ev[2].synchronize()
    fms = ev[0].elapsed_time(ev[1]) / k
    bms = ev[1].elapsed_time(ev[2]) / k
    es = 2 if cfg["dtype"] == wl.BF16 else 4
    V = cfg["V"]
    n_valid = int(((cfg["labels"] >= 0) & (cfg["labels"] < V)).sum())
    fbytes = n_valid * V * es + 12 * N
    bbytes = (2 * n_valid + (N - n_valid)) * V * es + 12 * N
    out.append({"path": "foak_ce_forward", "workload": WORKLOAD_DESC[args.workload], "steps": k, "ms_per_step": fms,
                "tokens_per_s": N / (fms * 1e-3), "GBps_algorithmic": fbytes / (fms * 1e-3) / 1e9,
                "frac": fbytes / (fms * 1e-3) / 1e9 / peak, "peak_source": peak_src})
    out.append({"path": "foak_ce_backward", "workload": WORKLOAD_DESC[args.workload], "steps": k,
                "ms_per_step": bms, "tokens_per_s": N / (bms * 1e-3),
                "GBps_algorithmic": bbytes / (bms * 1e-3) / 1e9, "frac": bbytes / (bms * 1e-3) / 1e9 / peak,
                "peak_source": peak_src})
    out.append({"path": "foak_ce_forward + foak_ce_backward", "workload": WORKLOAD_DESC[args.workload],
                "ms_per_step": fms + bms, "tokens_per_s": N / ((fms + bms) * 1e-3)})
    del bufs, dl
    torch.cuda.empty_cache()
    out.extend(chunked_timing(ce, torch, dev, stream))
    return out


CHUNKED_DESC = ("chunked linear+CE: H 8192x4096 bf16 ~N(0,1), W 32000x4096 bf16 ~N(0,0.02^2), 10% rows -100, "
                "chunks of 1024 rows")
ROPE_DESC = ("rotary embedding, Llama-3-8B attention shapes: Q 8192x32x128 and K 8192x8x128 bf16 ~N(0,1), "
             "packed sequences of up to 2048 tokens (position ids restart per sequence), base 500000")
NORM_TAIL_DESC = ("decoder tail: RMSNorm (eps 1e-5) of X 8192x4096 bf16 ~N(0,2^2), gamma ~N(1,0.1^2) -> "
                  "chunked LM head W 32000x4096 + CE, 10% rows -100, chunks of 1024 rows")


def chunked_timing(ce, torch, dev, stream, steps=10, warmup=3):
    """foak_linear_ce_chunked on the chunked workload, and its three GEMM shapes alone."""
    c = wl.chunked()
    N, V, D, chunk = c["N"], c["V"], c["D"], c["chunk"]
    H = torch.from_numpy(c["H"].view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(c["W"].view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.from_numpy(c["labels"]).to(dev)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, D, dtype=torch.float32, device=dev)
    peak, src = _peak_bf16(sustained=False)
    res = []

    def timed(fn, k, w):
        for _ in range(w):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / k

    def timed_graph(fn, k, w):
        """k calls captured in one CUDA graph, replayed once: the kernels' time without the
        host's per-call issue cost (a binding call costs ~15-20 us of Python, close to
        these kernels' own time)."""
        for _ in range(w):
            fn()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(graph):
                for _ in range(k):
                    fn()
        except RuntimeError as exc:  # no capture here: say so and time the calls eagerly
            print(f"graph capture failed ({exc}); timing eagerly", file=sys.stderr)
            return timed(fn, k, 0), "eager (graph capture failed)"
        graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        e1.synchronize()
        del graph
        return e0.elapsed_time(e1) / k, f"CUDA graph of {k} calls (host issue cost excluded)"

    ms = timed(lambda: ce.foak_linear_ce_chunked(H, W, y, chunk=chunk, dH=dH, dW=dW), steps, warmup)
    out = ce.foak_linear_ce_chunked(H, W, y, chunk=chunk, dH=dH, dW=dW)
    flops = 6.0 * N * V * D
    tf = flops / (ms * 1e-3) / 1e12
    res.append({"path": "foak_linear_ce_chunked", "workload": CHUNKED_DESC, "steps": steps, "ms_per_step": ms,
                "tokens_per_s": N / (ms * 1e-3), "TFLOPs": tf, "frac": tf / peak, "peak": peak,
                "peak_unit": "TFLOP/s bf16", "peak_source": src, "loss": float(out["loss"].item()),
                "err": int(out["err"].item()), "gpu_launches_per_step": 4 * ((N + chunk - 1) // chunk) + 1})
    # the decoder tail: final RMSNorm -> chunked LM head + CE -> norm backward
    t = wl.norm_chunked()
    X = torch.from_numpy(t["X"].view(np.int16)).to(dev).view(torch.bfloat16)
    gam = torch.from_numpy(t["gamma"].view(np.int16)).to(dev).view(torch.bfloat16)
    yt = torch.from_numpy(t["labels"]).to(dev)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    tail = lambda: ce.foak_rmsnorm_linear_ce_chunked(X, gam, W, yt, eps=t["eps"], chunk=chunk, dX=dX, dW=dW)  # noqa: E731
    ms_t = timed(tail, steps, warmup)
    out_t = tail()
    tf_t = flops / (ms_t * 1e-3) / 1e12
    res.append({"path": "foak_rmsnorm_linear_ce_chunked", "workload": NORM_TAIL_DESC, "steps": steps,
                "ms_per_step": ms_t, "tokens_per_s": N / (ms_t * 1e-3), "TFLOPs": tf_t, "frac": tf_t / peak,
                "peak": peak, "peak_unit": "TFLOP/s bf16 (6*N*V*D; the norm's bytes are not counted)",
                "peak_source": src, "norm_overhead_ms": ms_t - ms, "loss": float(out_t["loss"].item()),
                "err": int(out_t["err"].item())})
    # the norm alone, forward and backward (HBM-bound: algorithmic bytes / time)
    hbm, hsrc = _peak_hbm()
    Y = torch.empty_like(X)
    _, rstd = ce.foak_rmsnorm_forward(X, gam, eps=t["eps"], Y=Y)
    fwd = lambda: ce.foak_rmsnorm_forward(X, gam, eps=t["eps"], Y=Y)
    bwd = lambda: ce.foak_rmsnorm_backward(Y, X, gam, rstd, dX=dX)
    (ms_f, how_f), ms_fe = timed_graph(fwd, 20, 3), timed(fwd, 20, 3)
    (ms_b, how_b), ms_be = timed_graph(bwd, 20, 3), timed(bwd, 20, 3)
    nd2 = N * D * 2
    for name, ms_k, how, ms_e, byts in (("foak_rmsnorm_forward", ms_f, how_f, ms_fe, 2 * nd2 + 4 * N),
                                        ("foak_rmsnorm_backward (dX and dgamma)", ms_b, how_b, ms_be,
                                         3 * nd2 + 4 * N)):
        gbs = byts / (ms_k * 1e-3) / 1e9
        res.append({"path": name, "workload": "X 8192x4096 bf16 (the decoder tail's norm)", "steps": 20,
                    "ms_per_step": ms_k, "timing": how,
                    "ms_per_step_eager": ms_e, "GBps_algorithmic": gbs, "frac": gbs / hbm, "peak": hbm,
                    "peak_source": hsrc,
                    "bytes": "forward: read X, write Y; backward (one pass): read dY and X, write dX"})
    del X, dX, Y
    # rotary embedding on Llama-3-8B attention shapes (Q and K in place; HBM-bound)
    r = wl.rope_llama3()
    q = torch.from_numpy(r["Q"].view(np.int16)).to(dev).view(torch.bfloat16)
    k = torch.from_numpy(r["K"].view(np.int16)).to(dev).view(torch.bfloat16)
    pos = torch.from_numpy(r["positions"]).to(dev)
    cache = ce.foak_rope_cache(r["max_pos"], r["d"], base=r["base"], device=dev)

    def rope_step():
        ce.foak_rope_apply_qk(q, k, pos, cache)

    (ms_r, how_r), ms_re = timed_graph(rope_step, 20, 3), timed(rope_step, 20, 3)
    byts = 2 * (q.numel() + k.numel()) * 2 + 8 * pos.numel()
    gbs = byts / (ms_r * 1e-3) / 1e9
    res.append({"path": "foak_rope_apply_qk (Q and K in one launch, in place)", "workload": ROPE_DESC, "steps": 20,
                "ms_per_step": ms_r, "timing": how_r,
                "ms_per_step_eager": ms_re, "GBps_algorithmic": gbs, "frac": gbs / hbm, "peak": hbm, "peak_source": hsrc,
                "bytes": "Q and K read and written once, positions; the 4 MB cos/sin table stays in L2"})
    del q, k, cache
    # the products of the call at the shapes it runs them: a chunk's logits product and the
    # previous chunk's dH, alone and in the one grouped launch the call makes of them, and dW
    # once per group of four chunks
    G = 4
    Z = torch.empty(chunk, V, dtype=torch.bfloat16, device=dev)
    Zs = torch.randn(G * chunk, V, device=dev).to(torch.bfloat16)
    Hc = H[:chunk]
    Hg = H[:G * chunk]
    dHc = torch.empty(chunk, D, dtype=torch.bfloat16, device=dev)
    shapes = [
        ("Z = H_c W^T (M=1024, N=32000, K=4096, K/K-major)", chunk,
         lambda: ce.foak_gemm_bf16(Hc, W, Z, mode=ce.FOAK_GEMM_BF16)),
        ("dH_c = dZ W (M=1024, N=4096, K=32000, K/MN-major)", chunk,
         lambda: ce.foak_gemm_bf16(Zs[:chunk], W, dHc, b_mn_major=True, mode=ce.FOAK_GEMM_BF16)),
        ("Z(c) and dH(c-1) in one grouped launch (foak_gemm_bf16_group; the two shapes above)", 2 * chunk,
         lambda: ce.foak_gemm_bf16_group([dict(a=Hc, b=W, out=Z, mode=ce.FOAK_GEMM_BF16),
                                          dict(a=Zs[:chunk], b=W, out=dHc, b_mn_major=True,
                                               mode=ce.FOAK_GEMM_BF16)])),
        ("dW += dZ_g^T H_g (M=32000, N=4096, K=4096, MN/MN-major, fp32 TMA reduce-add of the 524 MB dW)",
         G * chunk,
         lambda: ce.foak_gemm_bf16(Zs, Hg, dW, a_mn_major=True, b_mn_major=True, mode=ce.FOAK_GEMM_F32_ACC)),
    ]
    for name, kk, fn in shapes:
        gms = timed(fn, 10, 3)
        gtf = 2.0 * kk * V * D / (gms * 1e-3) / 1e12
        res.append({"path": "foak_gemm_bf16", "workload": name, "steps": 10, "ms_per_step": gms, "TFLOPs": gtf,
                    "frac": gtf / peak, "peak_source": src})
    del H, W, dH, dW, Z, Zs
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- oracle legs

def _oracle_sample(cfg, rows, start=0):
    N = cfg["logits"].shape[0]
    idx = (np.arange(rows) + start) % N
    return np.ascontiguousarray(cfg["logits"][idx]), np.ascontiguousarray(cfg["labels"][idx])


def cpu_baseline(cfg, target_s=10.0):
    import oracle

    threads = oracle.default_threads()
    N = cfg["logits"].shape[0]
    done_rows, t = 0, 0.0
    start = 0
    rows = min(N, 256)
    while t < target_s:
        x, y = _oracle_sample(cfg, rows, start)
        t0 = time.perf_counter()
        oracle.ce(x, y, cfg["V"], threads=threads)
        t += time.perf_counter() - t0
        done_rows += rows
        start += rows
        if t < 0.5 * target_s and rows < N:
            rows = min(N, rows * 2)
    return {"value": done_rows / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done_rows} rows of the headline workload (consecutive rows, wrapping), float64 fwd+bwd "
                      f"incl. full gradient, {t:.1f} s"}


def run_reference(args, rank, world):
    import oracle

    cfg = _make(args.workload)
    threads = oracle.default_threads()
    N = cfg["logits"].shape[0]
    rows = 512  # per step: 32 rows per thread on 16 cores, so thread start-up does not dominate
    # distinct samples prepared before the timed region (their generation is not the oracle's work)
    pool = [_oracle_sample(cfg, rows, i * rows) for i in range(min(8, args.steps + args.warmup))]
    for i in range(args.warmup):
        x, y = pool[i % len(pool)]
        oracle.ce(x, y, cfg["V"], threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        x, y = pool[(args.warmup + i) % len(pool)]
        oracle.ce(x, y, cfg["V"], threads=threads)
    dt = time.perf_counter() - t0
    val = rows * args.steps / dt
    sample = (f"{rows} consecutive rows of the headline workload per step (N={N}; {len(pool)} distinct samples "
              "cycled), float64 fwd+bwd incl. gradient")
    return {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(cfg, args.workload),
            "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main

def _dp_module():
    """The data-parallel helpers, loaded without the package (the reference arm needs no library)."""
    import importlib.util

    path = os.path.join(ROOT, "cross_entropy_loss_gb300", "dp.py")
    spec = importlib.util.spec_from_file_location("_foak_dp", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESC), default="mistral")
    ap.add_argument("--quick", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--rows", type=int, default=0,
                    help="with --profile: keep only the first ROWS rows of the workload (smaller ncu captures)")
    ap.add_argument("--path", choices=["fused", "forward", "backward", "chunked"], default="fused",
                    help="with --profile: which entry point the timed loop calls")
    ap.add_argument("--profile", action="store_true",
                    help="headline timed loop only (no e2e, secondary, clocks or CPU baseline): for ncu captures")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    dp = _dp_module()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU (NCCL): start the ranks; rank 0 prints the line
        return dp.relaunch(args.gpus, os.path.abspath(__file__), sys.argv[1:])
    rank, world, local = dp.rank_env()
    dist = None
    if world > 1:
        if args.impl == "reference":
            if rank != 0:
                return 0
            print(json.dumps(run_reference(args, rank, 1)))
            return 0
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist

    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
