#!/usr/bin/env python
"""Benchmark of the chunked Gated DeltaNet forward + backward on GB300.

Metric: GDN chunk fwd+bwd tokens/s at T=4096, Hv=32, d=128 (one Qwen3-Next-
shaped GDN layer: B=1, 16 key heads shared by 32 value heads, chunk 128,
h0 ~ N(0, 0.1^2), g = -softplus(N(0,1) + 1), cotangents dO ~ N(0,1),
dhT ~ N(0, 0.1^2)), and the fraction of the binding roofline.

A step is one forward (o, hT) plus one backward (dq, dk, dv, dg, dbeta,
dh0) over one batch; the forward keeps its per-chunk w, u, P, T, states and
Delta for the backward (as a training step's autograd would), so the backward
runs only the reverse walk and the gradients.  Inputs are resident in HBM; L2 is flushed (a 512 MiB
write) before every timed step, outside the step's events.  The timed steps carry CUDA events only
around each whole step; the per-kernel split comes from a second pass of the same steps with an
event after every launch.  Each rank runs
the same per-GPU workload (weak scaling, no collective on the data path).

--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

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

# per-unit algorithmic work of the path (2 m n k per product, triangular
# operands at their nonzero size; K K^T and Q K^T once per key head)
def chunk_flops(C, D=128):
    """Per-chunk FLOPs at chunk size C: K K^T + Q K^T (per key head), the
    ladder (sum over its levels b = 1, 2, .., C/2 of 2 b^2 C), a lower-
    triangular C x C times C x D product, and a full C x D x D product."""
    ladder, b = 0, 1
    while b < C:
        ladder += 2 * b * b * C
        b *= 2
    return dict(khead=2 * C * C * D, ladder=ladder, tri=C * (C + 1) * D, full=2 * C * D * D)


_F128 = chunk_flops(128)
FLOP_PER_CHUNK_KHEAD = _F128["khead"]     # 4,194,304: K K^T + Q K^T (both triangular)
FLOP_LADDER = _F128["ladder"]             # 1,398,016: sum_b 2 b^2 C for b = 1..64
FLOP_TRI = _F128["tri"]                   # 2,113,536: lower-triangular 128x128 times 128x128
FLOP_FULL = _F128["full"]                 # 4,194,304: 128x128x128
FLOPS = {  # per (chunk, value head), per kernel
    "prep": FLOP_LADDER + 2 * FLOP_TRI,   # + FLOP_PER_CHUNK_KHEAD per (chunk, key head)
    "walk": 3 * FLOP_FULL + FLOP_TRI,     # w h, k_g^T Delta, Q h, P Delta
    "walk_states": 2 * FLOP_FULL,         # w h, k_g^T Delta
    "walk_bwd": 3 * FLOP_FULL + FLOP_TRI,  # K dh', Q^T dO, w^T dDelta, P^T dO
    "grads": 3 * FLOP_FULL + 9 * FLOP_TRI,
}
FLOPS["walks"] = FLOPS["walk_states"] + FLOPS["walk_bwd"]  # both walks of the backward, one launch
FWD_KERNELS = ["prep", "walk"]
FWD_KERNELS_SEG = ["prep", "fold", "prefix", "walk"]
# the backward of a step reads the w, u, P and T the forward kept (no preparation)
BWD_KERNELS = ["walk_bwd", "grads"]
BWD_KERNELS_SEG = ["fold_bwd", "prefix_bwd", "walk_bwd", "grads"]
KERNEL_SYMBOL = {"prep": "k_prep", "walk": "k_walk_fwd<0, 1, 32, 0>", "walks": "k_walk_pair", "grads": "k_grads",
                 "walk_bwd": "k_walk_bwd<0, 32>",
                 "fold": "k_walk_fwd<1, 0, 32, 0>", "prefix": "k_affine_walk",
                 "fold_bwd": "k_walk_bwd<1, 32>", "prefix_bwd": "k_affine_walk"}
# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum, bytes)
# from the committed ncu capture of the same kernel code (profiles/*), keyed by
# kernel; a kernel changed since its capture has no entry.
NCU_TRAFFIC = {"grads": 317395968}  # profiles/k_grads_layer_t4096_ncu_full.md: 270.86 MB + 46.54 MB


def algorithmic(wl):
    """Algorithmic bytes and FLOPs of the forward and backward at workload wl."""
    B, T, Hk, Hv, dk, dv = wl.B, wl.T, wl.Hk, wl.Hv, wl.dk, wl.dv
    NC = (T + wl.chunk - 1) // wl.chunk
    qk = 2 * B * T * Hk * dk * 2
    vv = B * T * Hv * dv * 2
    gb = 2 * B * T * Hv * 4
    st = B * Hv * dk * dv * 4
    fwd_bytes = qk + vv + gb + st + vv + st            # read q k v g beta h0, write o hT
    bwd_bytes = qk + vv + gb + st + vv + st + qk + vv + gb + st  # + dO dhT; dq dk dv dg dbeta dh0
    units, kunits = B * Hv * NC, B * Hk * NC
    f = chunk_flops(wl.chunk, dk)  # prep: ladder, w, u; walk: w h, k_g^T Delta, Q h, P Delta
    fwd_flops = kunits * f["khead"] + units * (f["ladder"] + 3 * f["tri"] + 3 * f["full"])
    # the backward takes w, u, P, T, the states and Delta from the forward: the
    # reverse walk and the chunk gradients
    bwd_flops = units * (FLOPS["walk_bwd"] + FLOPS["grads"])
    return dict(fwd_bytes=fwd_bytes, bwd_bytes=bwd_bytes, fwd_flops=fwd_flops,
                bwd_flops=bwd_flops, units=units, kunits=kunits)


def kernel_flops(name, alg):
    f = FLOPS.get(name)
    if f is None:
        return None
    extra = alg["kunits"] * FLOP_PER_CHUNK_KHEAD if name == "prep" else 0
    return alg["units"] * f + extra


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        return dict(hbm=float(mp["hbm_gbs"]), bf16=float(mp["bf16_tflops"]),
                    bf16_sustained=float(mp.get("bf16_tflops_sustained", mp["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "timed window"
        if not win:  # timed region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            win = [p for _, p in near]
            note = "nearest samples to a short timed window"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win), "window": note}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (ctypes, read-only
    queries) every millisecond, so that a timed region of a few milliseconds is
    still sampled many times.  Falls back silently when NVML is unavailable."""
    # clock-event reason bits (nvml.h): SW power cap, HW slowdown, SW thermal, HW thermal
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index, period_s=0.001):
        self.samples = []
        self.gpu = gpu_index
        self.period = period_s
        self.thread = None
        self.stop_flag = threading.Event()
        self.lib = None
        self.handle = None
        self.max_mhz = None

    def start(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        except (OSError, AttributeError):
            return
        self.lib, self.handle = lib, h
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        import ctypes
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            t = time.time()
            if self.lib.nvmlDeviceGetClockInfo(self.handle, ctypes.c_int(1), ctypes.byref(clk)) == 0:
                r = None
                if self.reasons_fn is not None and self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                    r = int(rs.value)
                self.samples.append((t, float(clk.value), r))
            time.sleep(self.period)

    def stop(self):
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        win = [x for x in self.samples if t0 <= x[0] <= t1]
        if not win:
            return None
        reasons = sorted({name for (_, _, r) in win if r is not None
                          for bit, name in self.BITS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for (_, m, _) in win), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(win),
                "window": "timed window, NVML every 1 ms"}


# ---------------------------------------------------------------- our arm
def kernel_table(kern, alg, pk, mean_step):
    """Per-kernel lines (mean ms per launch from CUDA events, share of the step,
    algorithmic TFLOP/s) and the roofline of the dominant kernel: its
    algorithmic FLOPs per launch over its mean launch time, against the
    measured bf16 peak, with the DRAM traffic of its ncu capture when the
    kernel is unchanged since.  Backward launches of a kernel carry "_b"."""
    kernels = {}
    for name, ms in kern.items():
        base = name[:-2] if name.endswith("_b") else name
        fl = kernel_flops(base, alg)
        kernels[name] = {"symbol": KERNEL_SYMBOL.get(base, base), "ms": round(ms, 5),
                         "share": round(ms / mean_step, 4)}
        if fl:
            kernels[name]["tflops"] = round(fl / (ms * 1e-3) / 1e12, 2)
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dbase = dom[:-2] if dom.endswith("_b") else dom
    dfl = kernel_flops(dbase, alg) or 0
    dms = kernels[dom]["ms"]
    achieved = dfl / (dms * 1e-3) / 1e12 if dfl else 0.0
    peak = pk["bf16"]
    roofline = {"kernel": KERNEL_SYMBOL.get(dbase, dbase), "bound": "tensor",
                "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": NCU_TRAFFIC.get(dom),
                "peak_source": f"bf16 burst, {pk['source']}",
                "timing": "mean launch time from CUDA events around each launch (the per-kernel pass)"}
    return kernels, roofline


def combine_ranks(total_ms, tokens_per_rank, world, rank, device=None):
    """Whole-job timing of `world` independent replicas: the slowest rank's
    timed span (a max over the process group when world > 1) and the tokens all
    ranks processed in it.  Returns (span_ms, tokens_per_s) on rank 0 and None
    on the other ranks, which print nothing."""
    import torch
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    if rank != 0:
        return None
    return total_ms, world * tokens_per_rank / (total_ms / 1e3)


def run_ours(args, rank, world, local_rank):
    import torch
    import linear_attention_rnn_gb300 as gdn
    from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gdn.build()
    wl = WORKLOADS[args.workload].replace(backward=True)
    nseg = args.n_segments if args.n_segments > 0 else gdn.default_segments(wl.B, wl.T, wl.Hv)
    host = make_host(wl)
    d = host.to(dev)
    ws_f = torch.empty(gdn.fwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg),
                       dtype=torch.uint8, device=dev)
    ws_b = torch.empty(gdn.bwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg),
                       dtype=torch.uint8, device=dev)
    sv = torch.empty(gdn.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    fk = FWD_KERNELS if nseg == 1 else FWD_KERNELS_SEG
    bk = BWD_KERNELS if nseg == 1 else BWD_KERNELS_SEG

    def mk_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record()
        return evs

    K, W = args.steps, args.warmup
    starts = mk_events(K)
    ends = mk_events(K)
    s_starts = mk_events(K)  # the per-kernel pass (events after every launch)
    fev = [mk_events(len(fk)) for _ in range(K)]
    bev = [mk_events(len(bk)) for _ in range(K)]
    torch.cuda.synchronize()

    def step(i=None):
        o, hT = gdn.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, n_segments=nseg, workspace=ws_f,
                              events=None if i is None else fev[i], saved=sv)
        gr = gdn.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, n_segments=nseg,
                           workspace=ws_b, events=None if i is None else bev[i], saved=sv)
        return o, hT, gr

    sampler = ClockSampler(local_rank)
    sampler.start()
    fast = NvmlSampler(local_rank)
    fast.start()
    # warm-up: at least W steps and at least ~1 s of device work
    t_w = time.time()
    n_w = 0
    while n_w < W or time.time() - t_w < args.min_warmup_s:
        flush.zero_()
        step()
        n_w += 1
        if n_w % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)  # head start for the host's launches
    # the timed steps: events only around each whole step (an event recorded
    # between two launches holds the second one back; measured 6 us per step)
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.stop()
    fast.stop()

    # the per-kernel split: the same K steps again, with an event after every launch
    for i in range(K):
        flush.zero_()
        s_starts[i].record()
        step(i)
    torch.cuda.synchronize()

    # the plain forward (gdn_chunk_fwd: o and hT only, nothing kept for a
    # backward), timed alone after the step's timed region
    plain = []
    for i in range(max(K, 10)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        gdn.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, n_segments=nseg, workspace=ws_f)
        e1.record()
        plain.append((e0, e1))
    torch.cuda.synchronize()
    fwd_plain_ms = statistics.median(a.elapsed_time(b) for a, b in plain)
    step_ms = [starts[i].elapsed_time(ends[i]) for i in range(K)]
    fwd_ms = [s_starts[i].elapsed_time(fev[i][-1]) for i in range(K)]
    bwd_ms = [fev[i][-1].elapsed_time(bev[i][-1]) for i in range(K)]
    kern = {}
    for name_list, evl, first in ((fk, fev, s_starts), (bk, bev, [f[-1] for f in fev])):
        for kidx, name in enumerate(name_list):
            key = name if name_list is fk else name + ("_b" if name in ("prep", "fold", "prefix") else "")
            ts = []
            for i in range(K):
                a = first[i] if kidx == 0 else evl[i][kidx - 1]
                ts.append(a.elapsed_time(evl[i][kidx]))
            kern[key] = sum(ts) / K
    total_ms = sum(step_ms)

    # e2e through the same public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, gdn, wl, host, dev, nseg)

    job = combine_ranks(total_ms, wl.tokens * K, world, rank, device=dev)
    if job is None:
        return None
    total_ms, value = job
    alg = algorithmic(wl)
    pk = peaks()
    mean_step = total_ms / K
    fwd_mean = statistics.mean(fwd_ms)
    bwd_mean = statistics.mean(bwd_ms)

    def path(bytes_, flops, ms):
        t_hbm = bytes_ / (pk["hbm"] * 1e9) * 1e3
        t_tc = flops / (pk["bf16"] * 1e12) * 1e3
        t_roof = max(t_hbm, t_tc)
        return {"ms": round(ms, 5), "roof_ms": round(t_roof, 5),
                "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": round(t_roof / ms, 4),
                "algorithmic_bytes": bytes_, "algorithmic_flops": flops}

    # shares of the per-kernel pass's own step (its events add about 6 us to a step)
    split_step = sum(kern.values())
    kernels, roofline = kernel_table(kern, alg, pk, split_step)
    clocks = fast.summary(t0, t1) or sampler.summary(t0, t1)
    clocks["nvidia_smi"] = {k: v for k, v in sampler.summary(t0, t1).items() if k != "window"}
    out = {
        "metric": "GDN chunk fwd+bwd tokens/s (T=4096, H_v=32, d=128) and % of roofline",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": n_w,
        "ms_per_step": round(mean_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{wl.name} fwd+bwd: B={wl.B} T={wl.T} Hk={wl.Hk} Hv={wl.Hv} "
                               f"dk=dv={wl.dk} chunk={wl.chunk} segments={nseg}",
                   "l2": "flushed (512 MiB write) before every timed step",
                   "parallelism": f"replicas x{world} (independent problems)"},
        "roofline": roofline,
        "path_roofline": {"fwd": path(alg["fwd_bytes"], alg["fwd_flops"], fwd_mean),
                          "fwd_plain": path(alg["fwd_bytes"], alg["fwd_flops"], fwd_plain_ms),
                          "bwd": path(alg["bwd_bytes"], alg["bwd_flops"], bwd_mean),
                          "step": path(alg["fwd_bytes"] + alg["bwd_bytes"],
                                       alg["fwd_flops"] + alg["bwd_flops"], mean_step),
                          "peaks": {"hbm_gbs": pk["hbm"], "bf16_tflops": pk["bf16"],
                                    "source": pk["source"]}},
        "kernels": kernels,
        "kernels_pass": {"how": "the K steps again, with a CUDA event after every launch",
                         "ms_per_step": round(split_step, 5)},
        "fwd_tokens_per_s": round(wl.tokens / (fwd_mean * 1e-3), 1),
        "bwd_tokens_per_s": round(wl.tokens / (bwd_mean * 1e-3), 1),
        "gpu_launches": K * (len(fk) + len(bk)),
        "clocks": clocks,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, host)
    return out


class Packed:
    """Tensors laid out in one byte buffer (each at a 256-byte-aligned offset),
    so that a step's inputs or results cross the host link in one copy."""

    def __init__(self, specs, device=None, pinned=False):
        import torch
        self.offsets, off = {}, 0
        for name, (shape, dtype) in specs.items():
            n = 1
            for x in shape:
                n *= x
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            self.offsets[name] = (off, nbytes, shape, dtype)
            off += (nbytes + 255) // 256 * 256
        self.nbytes = off
        self.buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pinned:
            self.buf = self.buf.pin_memory()
        self.views = {n: self.buf[o:o + nb].view(dt).view(shape)
                      for n, (o, nb, shape, dt) in self.offsets.items()}


def run_e2e(args, gdn, wl, host, dev, nseg):
    """Same step through the public API with pinned host buffers: every step
    copies its inputs host->device, runs forward + backward and copies every
    result device->host, all inside the timed region.  Steps are pipelined the
    way a training loop feeds a GPU: uploads, kernels and downloads run on
    three streams over two buffer sets, so step i+1's upload and step i-1's
    download overlap step i's kernels (events order each buffer's reuse).  A
    step's inputs sit in one packed buffer and its results are written into
    another, so each direction is a single copy (the host link carries one
    large copy faster than eight separate ones)."""
    import torch
    names_in = ["q", "k", "v", "g", "beta", "h0", "dO", "dhT"]
    spec_in = {n: (tuple(getattr(host, n).shape), getattr(host, n).dtype) for n in names_in}
    B, T, Hk, Hv, D = wl.B, wl.T, wl.Hk, wl.Hv, 128
    f32, b16 = torch.float32, torch.bfloat16
    spec_out = {"o": ((B, T, Hv, D), b16), "hT": ((B, Hv, D, D), f32),
                "dq": ((B, T, Hk, D), b16), "dk": ((B, T, Hk, D), b16), "dv": ((B, T, Hv, D), b16),
                "dg": ((B, T, Hv), f32), "dbeta": ((B, T, Hv), f32), "dh0": ((B, Hv, D, D), f32)}
    hin = Packed(spec_in, pinned=True)
    for n in names_in:
        hin.views[n].copy_(getattr(host, n))
    din = [Packed(spec_in, device=dev) for _ in range(2)]
    dout = [Packed(spec_out, device=dev) for _ in range(2)]
    hout = [Packed(spec_out, pinned=True) for _ in range(2)]
    ws_f = [torch.empty(gdn.fwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg),
                        dtype=torch.uint8, device=dev) for _ in range(2)]
    ws_b = [torch.empty(gdn.bwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg),
                        dtype=torch.uint8, device=dev) for _ in range(2)]
    svs = [torch.empty(gdn.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg), dtype=torch.uint8,
                       device=dev) for _ in range(2)]
    s_up, s_run, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up_done, run_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def one(i):
        k = i & 1
        with torch.cuda.stream(s_up):
            if i >= 2:
                s_up.wait_event(run_done[k])  # step i-2's kernels have read din[k]
            din[k].buf.copy_(hin.buf, non_blocking=True)
            up_done[k].record(s_up)
        with torch.cuda.stream(s_run):
            s_run.wait_event(up_done[k])
            if i >= 2:
                s_run.wait_event(down_done[k])  # step i-2's results have left dout[k]
            x, y = din[k].views, dout[k].views
            gdn.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], n_segments=nseg,
                          o=y["o"], hT=y["hT"], workspace=ws_f[k], saved=svs[k])
            gdn.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["dO"], x["dhT"],
                          n_segments=nseg, workspace=ws_b[k], saved=svs[k],
                          out=(y["dq"], y["dk"], y["dv"], y["dg"], y["dbeta"], y["dh0"]))
            run_done[k].record(s_run)
        with torch.cuda.stream(s_down):
            s_down.wait_event(run_done[k])
            hout[k].buf.copy_(dout[k].buf, non_blocking=True)
            down_done[k].record(s_down)

    for i in range(max(3, args.warmup)):
        one(i)
    torch.cuda.synchronize()
    K = args.steps
    # three timed runs of K steps: the host link and host memory are shared with
    # whatever else runs on the node, so the median is reported with the spread
    runs = []
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        for i in range(K):
            one(i)
        e1.record(s_down)  # after the last download, which follows every other step's work
        e1.synchronize()
        torch.cuda.synchronize()
        runs.append(e0.elapsed_time(e1))
    ms = statistics.median(runs)
    return {"value": round(wl.tokens * K / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": hin.nbytes, "d2h_bytes_per_step": dout[0].nbytes,
            "ms_per_step": round(ms / K, 5),
            "ms_per_step_runs": [round(r / K, 5) for r in runs], "reported": "median of 3 runs",
            "pipelined": "3 streams (upload, kernels, download), 2 buffer sets, one packed copy each way"}


# ---------------------------------------------------------------- oracle arm
def oracle_step(host, key_heads):
    """fp64 oracle forward + backward on the value heads of `key_heads`."""
    import oracle
    wl = host.wl
    grp = wl.Hv // wl.Hk
    heads = [(b, kh * grp + r) for b in range(wl.B) for kh in key_heads for r in range(grp)]
    oracle.fwd(host, heads=heads)
    oracle.bwd(host, heads=heads)


def cpu_baseline(wl, host, min_seconds=10.0, max_steps=30):
    """The fp64 oracle as it stands, timed on the host cores over whole steps of
    the workload (every value head, forward and backward) until at least
    `min_seconds` of work, after building it outside the timing."""
    import oracle
    oracle.lib()  # compiled and loaded outside the timing
    steps, t = 0, time.time()
    while True:
        oracle_step(host, list(range(wl.Hk)))
        steps += 1
        dt = time.time() - t
        if dt >= min_seconds or steps >= max_steps:
            break
    return {"value": round(wl.tokens * steps / dt, 2), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{steps} full {wl.name} fwd+bwd steps (all {wl.Hv} value heads), fp64, "
                      f"{dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host
    wl = WORKLOADS[args.workload].replace(backward=True)
    host = make_host(wl)
    oracle.build()
    # size each step so that warm-up + timed steps stay within ~2-3 minutes
    t = time.time()
    oracle_step(host, [0])
    per_kh = time.time() - t
    budget = 150.0 / max(1, args.steps + args.warmup)
    n_kh = max(1, min(wl.Hk, int(budget / max(per_kh, 1e-3))))
    kh = list(range(n_kh))
    for _ in range(max(0, args.warmup - 1)):
        oracle_step(host, kh)
    t = time.time()
    for _ in range(args.steps):
        oracle_step(host, kh)
    dt = time.time() - t
    frac = n_kh / wl.Hk
    value = wl.tokens * frac * args.steps / dt
    sample = (f"{n_kh} of {wl.Hk} key heads ({n_kh * wl.Hv // wl.Hk} of {wl.Hv} value heads) "
              f"of {wl.name} fwd+bwd per step, fp64; tokens scaled by that fraction")
    return {
        "impl": "reference",
        "metric": "GDN chunk fwd+bwd tokens/s (T=4096, H_v=32, d=128) and % of roofline",
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3 / frac, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl.name} fwd+bwd: B={wl.B} T={wl.T} Hk={wl.Hk} Hv={wl.Hv} "
                               f"dk=dv={wl.dk} chunk={wl.chunk}",
                   "l2": "n/a (host)", "parallelism": "host cores"},
        "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "sample": sample,
                         "value": round(value, 2)},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- all workloads
def run_sweep(args):
    """Times every workload (the five configurations plus the slow-decay
    reading of the million-token one) on one GPU: per workload, the median
    over timed steps of the forward (and backward where the workload has one),
    the per-kernel split from CUDA events after each launch (for segmented
    runs: prep, fold, prefix, replay walk), the whole-path roofline fraction,
    and the oracle's rate on a bounded sample.  Inputs are generated on the
    device and resident in HBM; L2 is flushed before every timed step.
    Prints one JSON line per workload."""
    import torch
    import linear_attention_rnn_gb300 as gdn
    import oracle
    from linear_attention_rnn_gb300.inputs import WORKLOADS, make_device, make_host

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    gdn.build()
    pk = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    names = []
    for spec in args.sweep.split(","):  # "all" stands for every workload as configured
        names += list(WORKLOADS) if spec == "all" else [spec]
    for spec in names:
        # "name" runs the workload as configured, "name@S" with S segments (0: the library's
        # choice); a "/64" suffix runs the forward alone with 64-token chunks
        base, _, ch = spec.partition("/")
        name, _, segs = base.partition("@")
        wl = WORKLOADS[name]
        if segs:
            wl = wl.replace(n_segments=int(segs))
        if ch:
            wl = wl.replace(chunk=int(ch), backward=wl.backward and int(ch) == 128)
        bwd = wl.backward
        C = wl.chunk
        nseg = wl.n_segments or gdn.default_segments(wl.B, wl.T, wl.Hv, C)
        big = wl.tokens > (1 << 16)
        steps = 5 if big else 20
        d = make_device(wl, dev)
        ws_f = torch.empty(gdn.fwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, chunk=C, n_segments=nseg),
                           dtype=torch.uint8, device=dev)
        ws_b = (torch.empty(gdn.bwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg),
                            dtype=torch.uint8, device=dev) if bwd else None)
        sv = (torch.empty(gdn.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=nseg), dtype=torch.uint8,
                          device=dev) if bwd else None)
        fk = FWD_KERNELS if nseg == 1 else FWD_KERNELS_SEG
        bk = BWD_KERNELS if nseg == 1 else BWD_KERNELS_SEG

        def evs(n):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            for x in e:
                x.record()
            return e
        start = [evs(1)[0] for _ in range(steps)]
        fev = [evs(len(fk)) for _ in range(steps)]
        bev = [evs(len(bk)) for _ in range(steps)] if bwd else None

        def step(i=None):
            gdn.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=C, n_segments=nseg, workspace=ws_f,
                          events=None if i is None else fev[i], saved=sv)
            if bwd:
                gdn.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, n_segments=nseg,
                              workspace=ws_b, events=None if i is None else bev[i], saved=sv)
        for _ in range(2 if big else 5):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        for i in range(steps):
            flush.zero_()
            start[i].record()
            step(i)
        torch.cuda.synchronize()
        fwd_ms = statistics.median(start[i].elapsed_time(fev[i][-1]) for i in range(steps))
        split = {}
        for kidx, kname in enumerate(fk):
            split[kname] = round(statistics.median(
                (start[i] if kidx == 0 else fev[i][kidx - 1]).elapsed_time(fev[i][kidx])
                for i in range(steps)), 5)
        alg = algorithmic(wl)

        def path(bytes_, flops, ms):
            t_hbm = bytes_ / (pk["hbm"] * 1e9) * 1e3
            t_tc = flops / (pk["bf16"] * 1e12) * 1e3
            t_roof = max(t_hbm, t_tc)
            return {"ms": round(ms, 5), "roof_ms": round(t_roof, 5),
                    "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": round(t_roof / ms, 4)}
        line = {"workload": spec, "B": wl.B, "T": wl.T, "Hk": wl.Hk, "Hv": wl.Hv, "chunk": C,
                "segments": nseg, "timed_steps": steps, "reported": "median",
                "fwd": path(alg["fwd_bytes"], alg["fwd_flops"], fwd_ms),
                "fwd_tokens_per_s": round(wl.tokens / (fwd_ms * 1e-3), 1),
                "fwd_kernels_ms": split}
        if bwd:
            bwd_ms = statistics.median(fev[i][-1].elapsed_time(bev[i][-1]) for i in range(steps))
            bsplit = {}
            for kidx, kname in enumerate(bk):
                bsplit[kname] = round(statistics.median(
                    (fev[i][-1] if kidx == 0 else bev[i][kidx - 1]).elapsed_time(bev[i][kidx])
                    for i in range(steps)), 5)
            line["bwd"] = path(alg["bwd_bytes"], alg["bwd_flops"], bwd_ms)
            line["bwd_kernels_ms"] = bsplit
            line["step_tokens_per_s"] = round(wl.tokens / ((fwd_ms + bwd_ms) * 1e-3), 1)
        # the oracle on a bounded sample: key head 0 (its value heads), at most
        # 65,536 tokens of batch row 0, forward (+ backward), scaled to tokens/s
        # of the whole workload
        ts = min(wl.T, 1 << 16)
        sub = make_host(wl.replace(B=1, T=ts, Hk=1, Hv=wl.Hv // wl.Hk, backward=bwd))
        oracle.lib()
        t = time.time()
        oracle.fwd(sub)
        if bwd:
            oracle.bwd(sub)
        dt = time.time() - t
        line["oracle"] = {"tokens_per_s": round(ts / dt / wl.Hk, 2), "cores": oracle.num_threads(),
                          "sample": f"key head 0 of {wl.Hk} ({wl.Hv // wl.Hk} value heads), "
                                    f"{ts} tokens, {'fwd+bwd' if bwd else 'fwd'}, {dt:.1f} s; "
                                    f"rate scaled by 1/{wl.Hk}"}
        print(json.dumps(line), flush=True)
        del d, ws_f, ws_b, sv
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_t4096")
    ap.add_argument("--n-segments", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up until this much wall time has passed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default=None,
                    help="time these workloads (comma-separated names, or 'all') instead of "
                         "the headline step; one JSON line per workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit at once
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl")
    try:
        out = run_ours(args, rank, world, local_rank)
        if out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
