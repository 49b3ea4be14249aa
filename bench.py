#!/usr/bin/env python
"""Attention-forward benchmark on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference]

A step is one ``attn_fwd`` call (the whole fused forward: tile schedule,
TMA loads, QK^T, masking, online softmax, rescale, PV, epilogue) over one
batch of the workload's synthetic inputs, resident in HBM.  The metric is
TFLOP/s under the convention 4*H*L^2*d per sequence, halved when causal.
L2 is flushed (256 MB write) before every timed step; each step is timed
with CUDA events on the launching stream.

Default workload: the ragged packed batch (16 sequences, L ~ U[256, 8192],
Hq 32, Hkv 8, d 128, causal, Q x4), the largest of the five workloads.  The
other four are timed briefly and reported under "per_workload".

Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
collective on the data path); value = FLOPs of all ranks / max rank time.

--impl reference runs the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores; rank 0
only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16) at 1 GB300; fraction of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAK = 1900.0       # TFLOP/s, used only when MEASURED_PEAKS.json is absent
FLUSH_BYTES = 256 << 20      # > 129 MB L2


# ------------------------------------------------------------------ distributed
def world() -> tuple:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, ws, _ = world()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, ws


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a float over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_rate(units_all_ranks: float, max_seconds: float) -> float:
    return units_all_ranks / max_seconds


# ------------------------------------------------------------------ helpers
def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except OSError:
        return {}


def kernel_source_hash(forward_only: bool = False) -> str:
    """Hash of the kernel sources (forward_only: without the backward's and
    the CUDA-core decode's headers, which define no forward kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_program_compilers_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if forward_only and name.startswith(("attn_bwd", "attn_decode_cc")):
            continue
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    ent = rec.get(workload_key)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash(forward_only=True):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm, mx, pw, reasons = [], [], [], set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ native arm
def run_workload(pkg, W, wl, seed, steps, warmup, dev, flush, sample_clocks=False):
    import torch
    inp = W.make_inputs(wl, seed)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    o = torch.empty_like(q)
    lse_shape = (wl.Hq, inp.n_arg) if wl.varlen else (wl.B, wl.Hq, wl.N)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    flops = W.causal_flops(wl, inp.lens)
    stream = torch.cuda.current_stream(dev)

    def step():
        pkg.attn_fwd(q, k, v, o, lse, wl.B, wl.Hq, wl.Hkv, inp.n_arg, wl.d, wl.scale,
                     wl.causal, cu, stream=stream.cuda_stream)

    for _ in range(warmup):
        flush.zero_()
        step()
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"device status after warm-up: {pkg.attn_status_string(st)}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if sample_clocks else None
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.__enter__()
    t0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    barrier()
    if sampler:
        sampler.__exit__(None, None, None)
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"device status after timing: {pkg.attn_status_string(st)}")
    per_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return dict(inp=inp, flops=flops, per_ms=per_ms, total_ms=sum(per_ms), wall_s=wall,
                clocks=sampler.summary() if sampler else None,
                tensors=(q, k, v, o, lse, cu), step=step)


# One exp2 per visible score; MUFU ex2 issues 32 lanes per clock per SM
# (measured on this GPU with a dependent-free ex2 loop), at the 2.07 GHz
# maximum SM clock on 152 SMs.
MUFU_EX2_PER_S = 32 * 152 * 2.07e9


def launch_floor_us(dev, flush):
    """CUDA-event time of the smallest kernel launch (a one-element fill),
    the floor under any launch of the short workloads.  Timed as the
    workloads are: behind the L2 flush, so that the launch is queued before
    the GPU reaches it and host overhead stays out of the interval."""
    import torch
    x = torch.empty(1, device=dev)
    for _ in range(10):
        x.zero_()
    ts = []
    for _ in range(30):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        a.record()
        x.zero_()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return round(statistics.median(ts), 2)


def dram_latency_us(pkg, dev, hops=20000, reps=3):
    """Latency of one load that misses the L2, from a one-thread pointer chase
    over a 512 MiB chain (tang, section 9.2: the latency term of the time
    floor); median of `reps` chases."""
    import torch
    scratch = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    result = torch.zeros(2, dtype=torch.int64, device=dev)
    ns = []
    for _ in range(reps):
        pkg.attn_probe_dram_latency(scratch, scratch.numel(), hops, result)
        torch.cuda.synchronize(dev)
        ns.append(int(result[0].item()) / hops)
    del scratch
    return round(statistics.median(ns) / 1e3, 4)


def work_units(wl, lens):
    """Work units (256 query rows of one sequence and head) a forward launch
    of this workload schedules: the W of the time floor's wave term."""
    return sum((L + 255) // 256 for L in lens) * wl.Hq


def secondary_rooflines(wl, rr, ms, hbm_gbs, floor_us, lat_us=None, peak=None, sms=152):
    """The bounds that matter for the short workloads: the minimum HBM bytes
    (Q, K, V read once, O and LSE written once) against the copy bandwidth,
    the exponentials (one per visible score, FLOPs / 4d) against the MUFU
    rate, the time against the launch floor, and the time floor of tang,
    section 9.2, read as
        T >= t_launch + max(t_lat + bytes / BW, flops / peak, ceil(W / W_res) t_lat)
    with W the launch's work units and W_res one per SM."""
    inp = rr["inp"]
    rows = inp.total_rows
    nbytes = rows * (2 * wl.Hq + 2 * wl.Hkv) * wl.d * 2 + rows * wl.Hq * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    ex2 = rr["flops"] / (4 * wl.d) / (ms / 1e3)
    out = {"us": round(ms * 1e3, 2), "launch_floor_us": floor_us, "min_bytes": nbytes,
           "hbm_gbs": round(gbs, 1),
           "frac_of_hbm": round(gbs / hbm_gbs, 4) if hbm_gbs else None,
           "exp2_per_s": float(f"{ex2:.4g}"), "frac_of_mufu": round(ex2 / MUFU_EX2_PER_S, 4)}
    if lat_us is not None and hbm_gbs and peak:
        waves = -(-work_units(wl, inp.lens) // sms)
        terms = {"lat_plus_bytes": lat_us + nbytes / (hbm_gbs * 1e9) * 1e6,
                 "flops": rr["flops"] / (peak * 1e12) * 1e6,
                 "waves_lat": waves * lat_us}
        floor = floor_us + max(terms.values())
        out.update({"dram_latency_us": lat_us, "waves": waves,
                    "time_floor_us": round(floor, 2),
                    "time_floor_terms_us": {k: round(v, 3) for k, v in terms.items()},
                    "x_floor": round(ms * 1e3 / floor, 2)})
    return out


def time_steps(step, steps, warmup, flush, stream):
    """CUDA-event times (ms) of `steps` calls of step(), L2 flushed before each."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s_.elapsed_time(e) for s_, e in zip(starts, ends)]


def run_window(pkg, dev, flush, steps):
    """Causal sliding window of 128 keys (tang, section 7.3's variant table:
    n = 8k, d = 64) against full causal attention on the same inputs; FLOPs
    count the visible (query, key) pairs only, 4 d per pair."""
    import torch
    B, H, N, d, Wn = 4, 16, 8192, 64, 128
    g = torch.Generator().manual_seed(2001)
    q, k, v = (torch.randn((B, N, H, d), generator=g).to(torch.bfloat16).to(dev)
               for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    win = lambda: pkg.attn_fwd_ex(q, k, v, o, lse, B, H, H, N, d, d ** -0.5, True,
                                  window=(Wn - 1, -1), stream=stream.cuda_stream)
    full = lambda: pkg.attn_fwd(q, k, v, o, lse, B, H, H, N, d, d ** -0.5, True,
                                stream=stream.cuda_stream)
    tw = statistics.median(time_steps(win, steps, 3, flush, stream))
    tf = statistics.median(time_steps(full, steps, 3, flush, stream))
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"window run: {pkg.attn_status_string(st)}")
    pairs = B * H * (Wn * N - Wn * (Wn - 1) // 2)
    return {"workload": f"sliding window {Wn} causal B{B} H{H} N{N} d{d}",
            "tflops": round(4 * d * pairs / (tw / 1e3) / 1e12, 2), "ms_per_step": round(tw, 5),
            "full_causal_ms_per_step": round(tf, 5)}


def run_decode(pkg, dev, flush, steps, hbm_gbs):
    """Decode step: one new query per sequence against full key/value caches
    (split keys + merge).  HBM-bound: GB/s of the bytes that must move (K, V
    caches read once, Q read, O and LSE written)."""
    import torch
    B, Hq, Hkv, d, Nk, Nq = 16, 32, 8, 128, 8192, 1
    g = torch.Generator().manual_seed(2002)
    q = torch.randn((B, Nq, Hq, d), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((B, Nk, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((B, Nk, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    n = pkg.attn_decode_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
    ws = torch.empty(((max(n, 16) + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: pkg.attn_fwd_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, d ** -0.5,
                                       False, None, ws, stream=stream.cuda_stream)
    t = statistics.median(time_steps(step, steps, 3, flush, stream))
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"decode run: {pkg.attn_status_string(st)}")
    nbytes = 2 * k.numel() * 2 + 2 * q.numel() * 2 + lse.numel() * 4
    gbs = nbytes / (t / 1e3) / 1e9
    return {"workload": f"decode B{B} Hq{Hq} Hkv{Hkv} d{d} Nq{Nq} Nk{Nk} (full caches)",
            "gbs": round(gbs, 1), "ms_per_step": round(t, 5), "bytes_per_step": nbytes,
            "frac_of_hbm": round(gbs / hbm_gbs, 4) if hbm_gbs else None,
            "workspace_bytes": n}


def run_decode_paged(pkg, dev, flush, steps, hbm_gbs, page_size=16):
    """The decode step of run_decode over paged caches: pages of page_size
    rows in a shuffled pool, addressed through a block table."""
    import torch
    B, Hq, Hkv, d, Nk, Nq = 16, 32, 8, 128, 8192, 1
    nb = Nk // page_size
    g = torch.Generator().manual_seed(2003)
    q = torch.randn((B, Nq, Hq, d), generator=g).to(torch.bfloat16).to(dev)
    kc = torch.randn((B * nb, page_size, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((B * nb, page_size, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    table = torch.randperm(B * nb, generator=g).to(torch.int32).reshape(B, nb).to(dev)
    sl = torch.full((B,), Nk, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    n = pkg.attn_decode_paged_workspace_bytes(B, Hq, Hkv, Nq, nb, page_size, d)
    ws = torch.empty(((max(n, 16) + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: pkg.attn_fwd_decode_paged(q, kc, vc, o, lse, B, Hq, Hkv, Nq, d, d ** -0.5,
                                             False, sl, table, nb, page_size, B * nb, ws,
                                             stream=stream.cuda_stream)
    t = statistics.median(time_steps(step, steps, 3, flush, stream))
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"paged decode run: {pkg.attn_status_string(st)}")
    nbytes = 2 * kc.numel() * 2 + 2 * q.numel() * 2 + lse.numel() * 4 + table.numel() * 4
    gbs = nbytes / (t / 1e3) / 1e9
    return {"workload": f"paged decode B{B} Hq{Hq} Hkv{Hkv} d{d} Nq{Nq} Nk{Nk} page {page_size} "
                        f"(shuffled pool)",
            "gbs": round(gbs, 1), "ms_per_step": round(t, 5), "bytes_per_step": nbytes,
            "frac_of_hbm": round(gbs / hbm_gbs, 4) if hbm_gbs else None}


BWD_SHAPES = {
    # the GQA prefill workload's shape; the kernels compute seven products of
    # the forward's size (S and dP recomputed in both kernels)
    "backward": (2, 32, 8, 4096, 128),
    # the long head-dim-256 prefill shape; three kernels (dV, dK, dQ) compute
    # sixteen products of the forward's per-block size
    "backward256": (1, 16, 2, 16384, 256),
    # the GQA prefill shape at head dim 64, through the two-kernel path and
    # through the single pass (five products; dQ by bulk reduce-adds)
    "backward64": (2, 32, 8, 4096, 64),
    "backward64_single": (2, 32, 8, 4096, 64),
}
BWD_SINGLE_PASS = {"backward64_single"}


def run_backward(pkg, dev, flush, steps, shape="backward", seqlen=None):
    """Backward (dQ, dK, dV from the forward's O and LSE), causal, of one of
    BWD_SHAPES (seqlen: another sequence length, for small profiling runs).
    TFLOP/s under the usual convention of 2.5x the forward's FLOPs (five
    products of the forward's size)."""
    import torch
    B, Hq, Hkv, N, d = BWD_SHAPES[shape]
    N = seqlen or N
    g = torch.Generator().manual_seed(2004)
    q = torch.randn((B, N, Hq, d), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16).to(dev)
    do = torch.randn((B, N, Hq, d), generator=g).to(torch.bfloat16).to(dev)
    o, lse = pkg.attention(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    single = shape in BWD_SINGLE_PASS
    n = (pkg.attn_bwd_single_pass_workspace_bytes if single else pkg.attn_bwd_workspace_bytes)(
        B, Hq, N)
    ws = torch.empty(((n + 15) // 16 * 4,), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    run = pkg.attn_bwd_single_pass if single else pkg.attn_bwd
    step = lambda: run(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, d ** -0.5, True,
                       workspace=ws, stream=stream.cuda_stream)
    t = statistics.median(time_steps(step, steps, 3, flush, stream))
    st = pkg.attn_get_status(stream.cuda_stream)
    if st != pkg.ATTN_OK:
        raise RuntimeError(f"backward run: {pkg.attn_status_string(st)}")
    fwd_flops = 4.0 * B * Hq * N * N * d / 2
    tf = 2.5 * fwd_flops / (t / 1e3) / 1e12
    peak = measured_peaks().get("bf16_tflops")
    return {"workload": f"backward B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} causal"
                        + (", single pass" if single else ""),
            "tflops": round(tf, 2), "ms_per_step": round(t, 5),
            "frac_of_peak": round(tf / peak, 4) if peak else None,
            "flop_convention": "2.5 x forward"}


def run_e2e(pkg, W, wl, inp, dev, steps):
    """Same metric through the public C ABI with host buffers: every step
    copies Q, K, V from pinned host memory, runs attn_fwd and reads O and LSE
    back to pinned host memory."""
    import torch
    qh, kh, vh = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
    q, k, v = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    o = torch.empty_like(q)
    lse_shape = (wl.Hq, inp.n_arg) if wl.varlen else (wl.B, wl.Hq, wl.N)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def step():
        q.copy_(qh, non_blocking=True)
        k.copy_(kh, non_blocking=True)
        v.copy_(vh, non_blocking=True)
        pkg.attn_fwd(q, k, v, o, lse, wl.B, wl.Hq, wl.Hkv, inp.n_arg, wl.d, wl.scale,
                     wl.causal, cu, stream=stream.cuda_stream)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms = e0.elapsed_time(e1)
    flops = W.causal_flops(wl, inp.lens)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return dict(ms=ms, steps=steps, flops=flops, h2d=h2d, d2h=d2h)


def run_e2e_pipelined(pkg, W, wl, inp, dev, steps):
    """The e2e measurement with step i+1's host-to-device copies and step i-1's
    device-to-host read overlapping step i's forward: two sets of device
    buffers and pinned host outputs, one stream each for the copies in, the
    forward and the copies out, ordered by events (a set is refilled only
    after its forward ran, an output set rewritten only after it was read
    back).  Every step still copies its own Q, K, V in and its O, LSE out;
    the interval runs from the first copy in to the last copy out."""
    import torch
    qh, kh, vh = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    lse_shape = (wl.Hq, inp.n_arg) if wl.varlen else (wl.B, wl.Hq, wl.N)
    sets = []
    for _ in range(2):
        q, k, v = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
        sets.append(dict(q=q, k=k, v=v, o=torch.empty_like(q),
                         lse=torch.empty(lse_shape, dtype=torch.float32, device=dev),
                         oh=torch.empty(q.shape, dtype=q.dtype).pin_memory(),
                         lh=torch.empty(lse_shape, dtype=torch.float32).pin_memory()))
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    ran = [None, None]     # forward of the set's last step done (inputs free)
    read = [None, None]    # read-back of the set's last step done (outputs free)

    def step(i):
        b = sets[i & 1]
        with torch.cuda.stream(s_in):
            if ran[i & 1] is not None:
                s_in.wait_event(ran[i & 1])
            b["q"].copy_(qh, non_blocking=True)
            b["k"].copy_(kh, non_blocking=True)
            b["v"].copy_(vh, non_blocking=True)
            loaded = ev()
            loaded.record(s_in)
        s_run.wait_event(loaded)
        if read[i & 1] is not None:
            s_run.wait_event(read[i & 1])
        pkg.attn_fwd(b["q"], b["k"], b["v"], b["o"], b["lse"], wl.B, wl.Hq, wl.Hkv, inp.n_arg,
                     wl.d, wl.scale, wl.causal, cu, stream=s_run.cuda_stream)
        done = ev()
        done.record(s_run)
        ran[i & 1] = done
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            b["oh"].copy_(b["o"], non_blocking=True)
            b["lh"].copy_(b["lse"], non_blocking=True)
            back = ev()
            back.record(s_out)
        read[i & 1] = back

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(s_in)
    for i in range(steps):
        step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    ms = e0.elapsed_time(e1)
    flops = W.causal_flops(wl, inp.lens)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sets[0]["oh"].numel() * 2 + sets[0]["lh"].numel() * 4
    return dict(ms=ms, steps=steps, flops=flops, h2d=h2d, d2h=d2h)


def run_e2e_one_copy_stream(pkg, W, wl, inp, dev, steps):
    """The e2e measurement with every copy on one copy stream, in the order
    in(0), in(1), out(0), in(2), out(1), ...: step i+1's inputs still go in
    while step i's forward runs, but the two directions never share the host
    link at the same time (on some hosts copies in and out that overlap each
    other move less than the two in turn).  Two buffer sets as in
    run_e2e_pipelined; the interval runs from the first copy in to the last
    copy out."""
    import torch
    qh, kh, vh = (t.pin_memory() for t in (inp.q, inp.k, inp.v))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    lse_shape = (wl.Hq, inp.n_arg) if wl.varlen else (wl.B, wl.Hq, wl.N)
    sets = []
    for _ in range(2):
        q, k, v = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
        sets.append(dict(q=q, k=k, v=v, o=torch.empty_like(q),
                         lse=torch.empty(lse_shape, dtype=torch.float32, device=dev),
                         oh=torch.empty(q.shape, dtype=q.dtype).pin_memory(),
                         lh=torch.empty(lse_shape, dtype=torch.float32).pin_memory()))
    s_copy, s_run = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    ran = [None, None]      # forward of the set's last step done (inputs free)
    loaded = [None, None]   # the set's inputs copied in
    read = [None, None]     # read-back of the set's last step done (outputs free)

    def copy_in(i):
        b = sets[i & 1]
        with torch.cuda.stream(s_copy):
            if ran[i & 1] is not None:
                s_copy.wait_event(ran[i & 1])
            b["q"].copy_(qh, non_blocking=True)
            b["k"].copy_(kh, non_blocking=True)
            b["v"].copy_(vh, non_blocking=True)
            e = ev()
            e.record(s_copy)
        loaded[i & 1] = e

    def forward_and_out(i, more):
        b = sets[i & 1]
        s_run.wait_event(loaded[i & 1])
        if read[i & 1] is not None:
            s_run.wait_event(read[i & 1])
        pkg.attn_fwd(b["q"], b["k"], b["v"], b["o"], b["lse"], wl.B, wl.Hq, wl.Hkv, inp.n_arg,
                     wl.d, wl.scale, wl.causal, cu, stream=s_run.cuda_stream)
        done = ev()
        done.record(s_run)
        ran[i & 1] = done
        if more:
            copy_in(i + 1)   # ahead of this step's read-back on the copy stream
        with torch.cuda.stream(s_copy):
            s_copy.wait_event(done)
            b["oh"].copy_(b["o"], non_blocking=True)
            b["lh"].copy_(b["lse"], non_blocking=True)
            back = ev()
            back.record(s_copy)
        read[i & 1] = back

    def run(n):
        copy_in(0)
        for i in range(n):
            forward_and_out(i, i + 1 < n)

    run(2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(s_copy)
    run(steps)
    e1.record(s_copy)
    torch.cuda.synchronize(dev)
    barrier()
    ms = e0.elapsed_time(e1)
    flops = W.causal_flops(wl, inp.lens)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sets[0]["oh"].numel() * 2 + sets[0]["lh"].numel() * 4
    return dict(ms=ms, steps=steps, flops=flops, h2d=h2d, d2h=d2h)


def cpu_baseline(W, wl, inp, target_s=12.0):
    """The fp64 oracle, as it stands, on a bounded seeded row sample of the
    same workload, timed on this host's cores."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()

    def rows_flops(rows):
        # 4*d per (query row, visible key) pair: the same convention as the GPU metric
        n = 0
        for (s, h, i) in rows:
            L = inp.lens[s]
            n += (i + 1) if wl.causal else L
        return 4.0 * wl.d * n

    def timed(rows):
        t0 = time.perf_counter()
        oracle.attn_fwd_oracle(inp.q, inp.k, inp.v, wl.B, wl.Hq, wl.Hkv, inp.n_arg, wl.d,
                               wl.scale, wl.causal, cu_seqlens=cu, rows=rows, nthreads=cores)
        return time.perf_counter() - t0

    probe = W.sample_rows(wl, inp.lens, 4)
    t = max(timed(probe), 1e-3)
    per_head = max(4, min(int(4 * target_s / t), max(inp.lens) * len(inp.lens)))
    rows = W.sample_rows(wl, inp.lens, per_head)
    t = timed(rows)
    f = rows_flops(rows)
    return {"value": f / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{per_head} seeded query rows per head x {wl.Hq} heads "
                      f"({len(rows)} rows, {f:.3e} FLOPs) of workload '{wl.name}', fp64, "
                      f"{t:.1f} s"}


def native(args):
    import torch
    import tensor_program_compilers_gb300 as pkg
    from tensor_program_compilers_gb300 import workloads as W

    rank, ws, local = world()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init("nccl")
    pkg.build()
    wl = W.BY_KEY[args.workload]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    res = run_workload(pkg, W, wl, wl.seed + rank, args.steps, args.warmup, dev, flush,
                       sample_clocks=(rank == 0))
    max_s = reduce_max(res["total_ms"] / 1e3, dev)
    flops_all = reduce_sum(res["flops"] * args.steps, dev)
    value = whole_job_rate(flops_all, max_s) / 1e12
    ms_per_step = max_s * 1e3 / args.steps

    peaks = measured_peaks()
    if "bf16_tflops" in peaks:
        peak, peak_src = float(peaks["bf16_tflops"]), "measured burst bf16 (MEASURED_PEAKS.json)"
    else:
        peak, peak_src = FALLBACK_PEAK, "fallback"
    avg_launch_s = res["total_ms"] / 1e3 / args.steps
    achieved = res["flops"] / avg_launch_s / 1e12
    traffic = recorded_traffic(args.workload)

    e2e = None
    if not args.no_e2e:
        r = run_e2e_pipelined(pkg, W, wl, res["inp"], dev, args.e2e_steps)
        e_max = reduce_max(r["ms"] / 1e3, dev)
        e_flops = reduce_sum(r["flops"] * r["steps"], dev)
        r1 = run_e2e_one_copy_stream(pkg, W, wl, res["inp"], dev, args.e2e_steps)
        o_max = reduce_max(r1["ms"] / 1e3, dev)
        rs = run_e2e(pkg, W, wl, res["inp"], dev, args.e2e_steps)
        s_max = reduce_max(rs["ms"] / 1e3, dev)
        # every schedule copies the same bytes in and out each step; the
        # headline is the fastest of the three measured here, all reported
        schedules = {
            "overlapped": {"value": whole_job_rate(e_flops, e_max) / 1e12,
                           "ms_per_step": e_max * 1e3 / r["steps"],
                           "how": "copies in of step i+1 and out of step i-1 overlap the "
                                  "forward of step i (three streams, two buffer sets)"},
            "one_copy_stream": {"value": whole_job_rate(reduce_sum(r1["flops"] * r1["steps"], dev),
                                                        o_max) / 1e12,
                                "ms_per_step": o_max * 1e3 / r1["steps"],
                                "how": "copies in and out on one copy stream (in of step i+1 "
                                       "ahead of out of step i), the forward on another"},
            "serial": {"value": whole_job_rate(reduce_sum(rs["flops"] * rs["steps"], dev),
                                               s_max) / 1e12,
                       "ms_per_step": s_max * 1e3 / rs["steps"],
                       "how": "copy in, forward, copy out in order on one stream"},
        }
        best = max(schedules, key=lambda k: schedules[k]["value"])
        e2e = {"value": schedules[best]["value"], "unit": UNIT,
               "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
               "steps": r["steps"], "ms_per_step": schedules[best]["ms_per_step"],
               "schedule": best, "how": schedules[best]["how"], "schedules": schedules}

    per_workload = {}
    if not args.no_per_workload:
        floor_us = launch_floor_us(dev, flush)
        lat_us = dram_latency_us(pkg, dev)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for key, other in W.BY_KEY.items():
            if key == args.workload:
                continue
            rr = run_workload(pkg, W, other, other.seed + rank, min(args.steps, 20), 3, dev, flush)
            ms = rr["total_ms"] / len(rr["per_ms"])
            tf = rr["flops"] / (ms / 1e3) / 1e12
            per_workload[key] = {"workload": other.name, "tflops": round(tf, 2),
                                 "ms_per_step": round(ms, 5), "frac_of_peak": round(tf / peak, 4),
                                 "median_ms": round(statistics.median(rr["per_ms"]), 5),
                                 "min_ms": round(min(rr["per_ms"]), 5),
                                 **secondary_rooflines(other, rr, ms, peaks.get("hbm_gbs"),
                                                       floor_us, lat_us, peak, sms)}
            del rr
        per_workload["window"] = run_window(pkg, dev, flush, min(args.steps, 20))
        per_workload["decode"] = run_decode(pkg, dev, flush, min(args.steps, 20),
                                            peaks.get("hbm_gbs"))
        per_workload["decode_paged"] = run_decode_paged(pkg, dev, flush, min(args.steps, 20),
                                                        peaks.get("hbm_gbs"))
        per_workload["backward"] = run_backward(pkg, dev, flush, min(args.steps, 20))
        per_workload["backward256"] = run_backward(pkg, dev, flush, min(args.steps, 10),
                                                   "backward256")
        for key in ("backward64", "backward64_single"):
            per_workload[key] = run_backward(pkg, dev, flush, min(args.steps, 20), key)

    base = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(W, wl, res["inp"], args.cpu_seconds)

    if rank == 0:
        inp = res["inp"]
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv,
                       "d": wl.d, "causal": wl.causal, "tokens": inp.total_rows,
                       "seq_lens": inp.lens if wl.varlen else wl.N,
                       "flops_per_step": res["flops"],
                       "l2": "flushed before every timed step (256 MB write)",
                       "parallelism": f"{ws} replica(s), each rank its own batch"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                         "peak_source": peak_src, "unit": UNIT,
                         "frac": round(achieved / peak, 4), "traffic": traffic},
            "cpu_baseline": base, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": res["clocks"],
            "kernel_ms": {"min": round(min(res["per_ms"]), 5),
                          "median": round(statistics.median(res["per_ms"]), 5)},
            "per_workload": per_workload,
        }
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ reference arm
def reference(args):
    rank, ws, _ = world()
    if rank != 0:
        return            # rank 0 alone runs the CPU reference
    import oracle
    from tensor_program_compilers_gb300 import workloads as W
    oracle.build()
    wl = W.BY_KEY[args.workload]
    inp = W.make_inputs(wl, wl.seed)
    cores = len(os.sched_getaffinity(0))
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    per_head = args.ref_rows_per_head
    rows = W.sample_rows(wl, inp.lens, per_head)
    f = 4.0 * wl.d * sum(((i + 1) if wl.causal else inp.lens[s]) for (s, h, i) in rows)

    def step():
        oracle.attn_fwd_oracle(inp.q, inp.k, inp.v, wl.B, wl.Hq, wl.Hkv, inp.n_arg, wl.d,
                               wl.scale, wl.causal, cu_seqlens=cu, rows=rows, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    value = f * args.steps / t / 1e12
    sample = (f"{per_head} seeded query rows per head x {wl.Hq} heads ({len(rows)} rows, "
              f"{f:.3e} FLOPs per step) of workload '{wl.name}', fp64")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": t * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                      "causal": wl.causal, "tokens": inp.total_rows},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["ragged", "gqa", "d256", "block", "tiny"],
                    default="ragged")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--bwd-seqlen", type=int, default=None,
                    help="with --extra backward*: another sequence length (profiling)")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows-per-head", type=int, default=24)
    ap.add_argument("--extra", choices=["window", "decode", "decode_paged", *BWD_SHAPES],
                    default=None,
                    help="time only this extra path (one JSON line; for profiling)")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def extra_only(args):
    import torch
    import tensor_program_compilers_gb300 as pkg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkg.build()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    if args.extra == "window":
        out = run_window(pkg, dev, flush, args.steps)
    elif args.extra in BWD_SHAPES:
        out = run_backward(pkg, dev, flush, args.steps, args.extra, args.bwd_seqlen)
    elif args.extra == "decode_paged":
        out = run_decode_paged(pkg, dev, flush, args.steps, measured_peaks().get("hbm_gbs"))
    else:
        out = run_decode(pkg, dev, flush, args.steps, measured_peaks().get("hbm_gbs"))
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.extra:
        extra_only(args)
    elif args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
