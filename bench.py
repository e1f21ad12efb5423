#!/usr/bin/env python3
"""Throughput of multi-head scaled dot-product attention, forward + backward, on GB300.

One step = attn_fwd followed by attn_bwd (the whole path: O, lse, dQ, dK, dV)
over one synthetic batch of the chosen workload, inputs resident in HBM.
Default workload: the largest single-GPU training configuration, B=4, h=16,
n=m=16384, d_k=d_v=128, non-causal (long-sequence training; the paper's
O(n^2 d) cost per layer, §4 and Table 1, is what this shape stresses). The
short-sequence configurations of the base and big models are in the sweep.

metric: attention TFLOPS (bf16, fwd and bwd) with the FLOP convention
4*B*h*n*m*d_k for the forward (halved when causal) and 2.5x that for the
backward (five GEMMs), i.e. 3.5 * 4*B*h*n*m*d_k per step.

Multi-GPU (torchrun): every rank runs its own batch (the heads are
independent problems, §3.2.2); no collective touches the data path.
``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from seeded_inputs import WORKLOADS, Workload, kv_lengths  # noqa: E402

METRIC = "attention TFLOPS (bf16, fwd and bwd) and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
DEFAULT_WORKLOAD = "long_n16384_d128_nc"
# L2 size used to size the rotating input sets. The same number on every arm
# and box keeps `config` identical between the two arms; the GPU arm checks
# that the sets exceed twice the device's real L2.
NOMINAL_L2_BYTES = 136 * 10**6
CSRC = os.path.join(ROOT, "transformer_scaled_dot_attn_gb300", "csrc")


def step_flops(w: Workload) -> float:
    return w.fwd_flops() + w.bwd_flops()


def input_sets(w: Workload, l2_bytes: int = NOMINAL_L2_BYTES):
    """(number of rotating input sets, bytes of one set): Q, K, V, dO of the
    batch; enough sets that their total exceeds twice the L2."""
    set_bytes = 2 * (2 * w.heads * w.n * w.d_k + 2 * w.heads * w.m * w.d_k)
    n_sets = max(2, min(64, math.ceil(2 * l2_bytes / max(set_bytes, 1)) + 1))
    return n_sets, set_bytes


def workload_config(w: Workload, world: int) -> dict:
    n_sets, set_bytes = input_sets(w)
    return {"workload": f"{w.name}: B={w.B}, h={w.h}, n={w.n}, m={w.m}, d_k=d_v={w.d_k}, "
                        f"causal={w.causal}" + (f", Q x {w.q_mult:g}" if w.q_mult != 1 else "")
                        + (f", window={w.window}" if w.window is not None else ""),
            "global_batch": w.B * world, "seq_len": w.n, "kv_len": w.m, "heads": w.h,
            "head_dim": w.d_k, "causal": w.causal,
            "parallelism": f"replicas x{world} (independent batches)", "step": "attn_fwd + attn_bwd",
            "l2": f"inputs larger than L2: {n_sets} rotating input sets of {set_bytes / 1e6:.0f} MB"}


def whole_head_backward(w: Workload) -> bool:
    """True where the library runs the single-launch whole-head backward (it needs no workspace)."""
    import transformer_scaled_dot_attn_gb300 as A
    return A.attn_bwd_workspace_bytes(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal) == 0


def kernel_model(w: Workload):
    """Algorithmic FLOPs and bytes per launch of the two tensor-core kernels.

    fwd:      reads Q, K, V (bf16); writes O (bf16) and lse (fp32).
    bwd_main: general path: reads Q, dO, K, V (bf16) and the two fp32 row
              statistics; writes dK, dV (bf16) and the fp32 dQ accumulator once.
              Whole-head path (n <= 256, d <= 64): reads Q, dO, O, K, V (bf16)
              and lse (fp32); writes dQ, dK, dV (bf16).
    """
    H, n, m, d = w.heads, w.n, w.m, w.d_k
    fwd_bytes = H * (2 * (2 * n * d + 2 * m * d) + 4 * n)
    if whole_head_backward(w):
        bwd_bytes = H * (2 * (3 * n * d + 2 * m * d) + 4 * n + 2 * (n * d + 2 * m * d))
    else:
        bwd_bytes = H * (2 * (2 * n * d + 2 * m * d) + 8 * n + 2 * (2 * m * d) + 4 * n * d)
    return {
        "fwd": {"flops": w.fwd_flops(), "bytes": fwd_bytes},
        "bwd_main": {"flops": w.bwd_flops(), "bytes": bwd_bytes},
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# Sources of each kernel whose DRAM traffic is recorded: its own file and the
# device headers every kernel includes.
KERNEL_HEADERS = ("attn_kernels.cuh", "sm103_ptx.cuh")


def kernel_source_hash(files) -> str:
    """Hash of the given kernel sources (file names under csrc/)."""
    h = hashlib.sha256()
    for f in sorted(set(files) | set(KERNEL_HEADERS)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if that kernel's sources are unchanged."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    rec = d.get(workload, {}).get(kernel)
    if not rec or not rec.get("sources") or rec.get("source_hash") != kernel_source_hash(rec["sources"]):
        return None
    return rec.get("bytes_per_launch")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 20 ms) around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float, margin: float = 0.25):
        rows = []
        for ts, line in self.samples:
            if t0 - margin <= ts <= t1 + margin:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ----------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def _reduce(x: float, op_name: str) -> float:
    import torch
    import torch.distributed as dist
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=getattr(dist.ReduceOp, op_name))
    return float(t.item())


def reduce_max(x: float, world: int) -> float:
    """Max over ranks (the slowest rank's time bounds the whole job)."""
    return x if world == 1 else _reduce(x, "MAX")


def reduce_sum(x: float, world: int) -> float:
    """Sum over ranks (units of work processed by all ranks)."""
    return x if world == 1 else _reduce(x, "SUM")


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle sample

def visible_keys(w: Workload, i: int) -> int:
    """Keys that query row i of a head sees (no key padding): causal mask and window."""
    hi = w.m
    if w.causal:
        hi = min(hi, i + 1)
    lo = 0
    if w.window is not None:
        wl, wr = w.window
        if wr >= 0:
            hi = min(hi, i + wr + 1)
        if wl >= 0:
            lo = max(0, i - wl)
    return max(0, hi - lo)


def oracle_sample(w: Workload, target_s: float):
    """Time the fp64 oracle on a bounded sample of ``w``, about ``target_s`` seconds of CPU work.

    Whole heads (forward + backward, the step's FLOP convention) while one head
    takes under half of ``target_s``; otherwise evenly spaced query rows of the
    first head: their forward rows (O, lse) and their dQ rows, counted as
    4*d FLOPs per visible key for the forward row and 6*d for the dQ row (the
    score recomputation, dP and dQ: three of the backward's five products).
    Returns (TFLOP/s, seconds, sample description, threads).
    """
    import oracle
    from seeded_inputs import workload_inputs
    oracle.build()
    scale = w.default_scale
    q1, k1, v1, do1 = (t[0, 0] for t in workload_inputs(w, with_grad=True, heads=1))

    def run_rows(rows):
        t0 = time.perf_counter()
        oracle.fwd(q1, k1, v1, w.causal, scale, rows=rows, window=w.window)
        oracle.bwd_rows(q1, k1, v1, do1, w.causal, scale, qrows=rows, window=w.window)
        return time.perf_counter() - t0

    def rows_flops(rows):
        return sum(10.0 * w.d_k * visible_keys(w, i) for i in rows)

    def spaced(r):
        r = max(1, min(w.n, r))
        return sorted({int(i * w.n / r) for i in range(r)})

    rows = spaced(8)
    run_rows(rows)  # the first call pays one-time costs (library load, thread start)
    t = run_rows(rows)
    while t < 0.25 and len(rows) < w.n:
        rows = spaced(len(rows) * 4)
        t = run_rows(rows)
    rate = rows_flops(rows) / max(t, 1e-9)
    per_head = step_flops(w) / w.heads
    if per_head / rate <= target_s / 2:
        def run(heads):
            q, k, v, do = workload_inputs(w, with_grad=True, heads=heads)
            t0 = time.perf_counter()
            oracle.bwd(q, k, v, do, w.causal, scale, window=w.window)
            return time.perf_counter() - t0

        heads = max(1, min(w.heads, int(target_s / max(per_head / rate, 1e-9))))
        t = run(heads)
        return (per_head * heads / t / 1e12, t,
                f"{heads} of {w.heads} heads of {w.name}, forward and backward, {t:.1f} s", oracle.num_threads())
    rows = spaced(int(len(rows) * target_s / max(t, 1e-9)))
    t = run_rows(rows)
    return (rows_flops(rows) / t / 1e12, t,
            f"{len(rows)} of {w.n} query rows (evenly spaced) of one of {w.heads} heads of {w.name}: "
            f"forward rows and dQ rows, {t:.1f} s", oracle.num_threads())


# ----------------------------------------------------------------- GPU arm

def make_inputs(w: Workload, seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = (torch.randn(w.B, w.h, w.n, w.d_k, device=device, generator=g) * w.q_mult).bfloat16()
    k = torch.randn(w.B, w.h, w.m, w.d_k, device=device, generator=g).bfloat16()
    v = torch.randn(w.B, w.h, w.m, w.d_v, device=device, generator=g).bfloat16()
    do = torch.randn(w.B, w.h, w.n, w.d_v, device=device, generator=g).bfloat16()
    return q, k, v, do


def run_gpu(args, w: Workload, world, rank, local):
    import torch
    import transformer_scaled_dot_attn_gb300 as A

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    A.load_library()
    scale = w.default_scale
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets, set_bytes = input_sets(w)
    if n_sets * set_bytes <= 2 * l2:
        raise RuntimeError(f"input sets ({n_sets} x {set_bytes} B) do not exceed twice the L2 ({l2} B)")
    sets = [make_inputs(w, 1000 * rank + 17 * s + w.cfg, dev) for s in range(n_sets)]
    o = torch.empty(w.B, w.h, w.n, w.d_v, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.h, w.n, dtype=torch.float32, device=dev)
    dq = torch.empty(w.B, w.h, w.n, w.d_k, dtype=torch.bfloat16, device=dev)
    dk = torch.empty(w.B, w.h, w.m, w.d_k, dtype=torch.bfloat16, device=dev)
    dv = torch.empty(w.B, w.h, w.m, w.d_v, dtype=torch.bfloat16, device=dev)
    ws_bytes = A.attn_bwd_workspace_bytes(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    lens = kv_lengths(w)  # key padding of a variable-length workload (None: none)
    kvl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)

    def step(i):
        q, k, v, do = sets[i % n_sets]
        A.attn_fwd(q, k, v, causal=w.causal, scale=scale, out=o, lse=lse, kv_len=kvl, window=w.window)
        A.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=scale, dq=dq, dk=dk, dv=dv,
                   workspace=ws, kv_len=kvl, window=w.window)

    # settle clocks, then the counted warm-up
    t_soak = time.time()
    i = 0
    while time.time() - t_soak < args.soak_seconds:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if A.attn_get_device_status() != A.ATTN_OK:
        raise RuntimeError("device watchdog fired during warm-up")

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    A.attn_profile_enable(True)
    for kind in A.KERNEL_KINDS:
        A.attn_profile_read(kind)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    A.attn_profile_enable(False)
    ms = start.elapsed_time(end)
    prof = {kind: A.attn_profile_read(kind) for kind in A.KERNEL_KINDS}
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    status = A.attn_get_device_status()
    if status != A.ATTN_OK:
        raise RuntimeError(f"device status {A.attn_status_string(status)} in the timed region")
    launches = sum(n for n, _ in prof.values())

    ms_max = reduce_max(ms, world)
    total_flops = reduce_sum(step_flops(w) * args.steps, world)
    value = total_flops / (ms_max / 1e3) / 1e12

    # ---- end to end: pinned host inputs -> device -> fwd+bwd -> O, dQ, dK, dV back to host.
    # The library's host-buffer step (attn_fwd_bwd_host) splits the heads into
    # chunks whose copies in both directions overlap the kernels; the plain
    # sequence (all inputs in, fwd, bwd, all results out, one stream) is timed
    # beside it. Masked workloads (key padding, windows) have no host step.
    hq, hk, hv, hdo = [t.cpu().pin_memory() for t in sets[0]]
    d_in = [torch.empty_like(t) for t in sets[0]]
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, dq, dk, dv)]
    e2e_steps = max(1, min(args.steps, 20))
    host_step = kvl is None and w.window is None
    hbuf = A.HostStepBuffers(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal, device=dev) if host_step else None

    def e2e_serial():
        for dst, src in zip(d_in, (hq, hk, hv, hdo)):
            dst.copy_(src, non_blocking=True)
        A.attn_fwd(d_in[0], d_in[1], d_in[2], causal=w.causal, scale=scale, out=o, lse=lse, kv_len=kvl,
                   window=w.window)
        A.attn_bwd(d_in[0], d_in[1], d_in[2], o, lse, d_in[3], causal=w.causal, scale=scale,
                   dq=dq, dk=dk, dv=dv, workspace=ws, kv_len=kvl, window=w.window)
        for dst, src in zip(outs_h, (o, dq, dk, dv)):
            dst.copy_(src, non_blocking=True)

    def e2e_pipelined():
        A.attn_fwd_bwd_host(hq, hk, hv, hdo, causal=w.causal, scale=scale, buffers=hbuf, chunks=args.chunks,
                            out=(outs_h[0], None, outs_h[1], outs_h[2], outs_h[3]), stream=stream)

    def time_e2e(fn):
        fn()
        torch.cuda.synchronize()
        barrier(world)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(e2e_steps):
            fn()
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(s2.elapsed_time(e2), world)
        return reduce_sum(step_flops(w) * e2e_steps, world) / (e2e_ms / 1e3) / 1e12

    serial_value = time_e2e(e2e_serial)
    e2e_value = time_e2e(e2e_pipelined) if host_step else serial_value
    if A.attn_get_device_status() != A.ATTN_OK:
        raise RuntimeError("device watchdog fired in the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in outs_h)

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    model = kernel_model(w)
    kinds = {"fwd": prof["fwd"], "bwd_main": prof["bwd_main"]}
    dom = max(kinds, key=lambda k: kinds[k][1])
    n_launch, tot_ms = kinds[dom]
    avg_s = tot_ms / max(n_launch, 1) / 1e3
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = model[dom]["flops"] / model[dom]["bytes"]
    if intensity < ridge:
        achieved = model[dom]["bytes"] / avg_s / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "unit": "GB/s"}
    else:
        achieved = model[dom]["flops"] / avg_s / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "unit": "TFLOP/s"}
    roof.update({"kernel": dom, "achieved": round(achieved, 2), "peak": peak,
                 "peak_source": peak_src, "frac": round(achieved / peak, 4),
                 "traffic": recorded_traffic(dom, w.name),
                 "algorithmic_bytes": model[dom]["bytes"], "algorithmic_flops": model[dom]["flops"],
                 "avg_launch_us": round(avg_s * 1e6, 2)})
    per_kernel = {k: {"launches": n, "avg_us": round(t / max(n, 1) * 1e3, 2)} for k, (n, t) in prof.items()
                  if n > 0}
    for k in ("fwd", "bwd_main"):
        n_, t_ = prof[k]
        a = t_ / max(n_, 1) / 1e3
        per_kernel[k]["tflops"] = round(model[k]["flops"] / a / 1e12, 1) if n_ else None
        per_kernel[k]["gbs"] = round(model[k]["bytes"] / a / 1e9, 1) if n_ else None
    clocks = sampler.summary(t0, t1) if sampler else None
    return {
        "value": value, "ms_per_step": ms_max / args.steps, "launches": launches,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "attn_fwd_bwd_host" if host_step else "attn_fwd + attn_bwd",
                "chunks": args.chunks if host_step else None,
                "serial_value": round(serial_value, 3)},
        "roofline": roof, "kernels": per_kernel, "clocks": clocks, "n_sets": n_sets,
        "l2_bytes": l2, "set_bytes": set_bytes, "peaks": peaks,
    }


def run_sweep(args, local):
    """Per-configuration throughput of attn_fwd and attn_bwd (rank 0, N=1 only).

    Every case rotates input sets whose total exceeds twice the L2, and takes
    the median over 5 repeats of at least 10 steps each (at least 50 steps and
    200 ms per case); the times are the library's per-kernel CUDA events on the
    launching stream.
    """
    import torch
    import transformer_scaled_dot_attn_gb300 as A
    dev = torch.device("cuda", local)
    peaks, _ = load_peaks()
    out = {}
    names = ["encoder", "encoder_sat", "encoder_kpad", "decoder", "cross", "cross_h4_d128", "cross_h16_d32"]
    names += [f"long_n{n}_d{d}_{c}" for n in (1024, 4096, 16384) for d in (64, 128) for c in ("nc", "c")]
    names += ["long_n16384_d64_band257", "long_n16384_d64_local256"]
    for name in names:
        w = WORKLOADS[name]
        n_sets, _ = input_sets(w)
        sets = [make_inputs(w, 99 + 7 * i, dev) for i in range(n_sets)]
        lens = kv_lengths(w)
        kvl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
        kw = dict(causal=w.causal, scale=w.default_scale, kv_len=kvl, window=w.window)
        o, lse = A.attn_fwd(*sets[0][:3], **kw)
        dq, dk, dv = A.attn_bwd(*sets[0][:3], o, lse, sets[0][3], **kw)
        ws_bytes = A.attn_bwd_workspace_bytes(w.B, w.h, w.n, w.m, w.d_k, w.d_v, w.causal)
        ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

        def step(i):
            q, k, v, do = sets[i % n_sets]
            A.attn_fwd(q, k, v, out=o, lse=lse, **kw)
            A.attn_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, **kw)

        t0 = time.perf_counter()
        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        est = (time.perf_counter() - t0) / 3
        per_rep = max(10, math.ceil(0.04 / max(est, 1e-6)))
        f_list, b_list = [], []
        for rep in range(5):
            A.attn_profile_enable(True)
            for kind in A.KERNEL_KINDS:
                A.attn_profile_read(kind)
            for i in range(per_rep):
                step(i)
            torch.cuda.synchronize()
            A.attn_profile_enable(False)
            prof = {kind: A.attn_profile_read(kind) for kind in A.KERNEL_KINDS}
            f_list.append(prof["fwd"][1] / max(prof["fwd"][0], 1))
            b_list.append(sum(prof[kd][1] for kd in ("bwd_pre", "bwd_main", "bwd_post")) /
                          max(prof["bwd_main"][0], 1))
        f_ms, b_ms = statistics.median(f_list), statistics.median(b_list)
        ftf = w.fwd_flops() / (f_ms / 1e3) / 1e12
        btf = w.bwd_flops() / (b_ms / 1e3) / 1e12
        out[name] = {"fwd_us": round(f_ms * 1e3, 1), "fwd_tflops": round(ftf, 1),
                     "fwd_frac_peak": round(ftf / peaks["bf16_tflops"], 3),
                     "bwd_us": round(b_ms * 1e3, 1), "bwd_tflops": round(btf, 1),
                     "bwd_frac_peak": round(btf / peaks["bf16_tflops"], 3),
                     "steps": 5 * per_rep, "input_sets": n_sets}
        del sets, o, lse, dq, dk, dv, kvl, ws
        torch.cuda.empty_cache()
    if A.attn_get_device_status() != A.ATTN_OK:
        raise RuntimeError("device watchdog fired in the sweep")
    return out


def run_decode_sweep(args, local):
    """Throughput of one decoding step (attn_decode, split keys + merge) per decoding workload.

    HBM-bound: bytes = the caches K and V read once (B*h*m*d*2 each) plus q and
    o; FLOPs = 4*d per visible (query, key) pair. Rank 0, N=1 only.
    """
    import torch
    import transformer_scaled_dot_attn_gb300 as A
    from seeded_inputs import DECODE_WORKLOADS
    dev = torch.device("cuda", local)
    peaks, _ = load_peaks()
    out = {}
    for name, (B, h, n, m, d) in DECODE_WORKLOADS.items():
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        # inputs larger than L2: rotate enough cache copies between steps
        one = 2 * B * h * m * d * 2
        nsets = max(1, min(4, -(-3 * (129 << 20) // one)))
        sets = [(torch.randn(B, h, n, d, device=dev, generator=g).bfloat16(),
                 torch.randn(B, h, m, d, device=dev, generator=g).bfloat16(),
                 torch.randn(B, h, m, d, device=dev, generator=g).bfloat16()) for _ in range(nsets)]
        ws = torch.empty(A.attn_decode_workspace_bytes(B, h, n, m, d, d) // 4 + 4, dtype=torch.float32, device=dev)
        o = torch.empty(B, h, n, d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, h, n, dtype=torch.float32, device=dev)
        for i in range(3):
            A.attn_decode(*sets[i % nsets], out=o, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        iters = 40
        A.attn_profile_enable(True)
        for kind in A.KERNEL_KINDS:
            A.attn_profile_read(kind)
        for i in range(iters):
            A.attn_decode(*sets[i % nsets], out=o, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        A.attn_profile_enable(False)
        c1, ms1 = A.attn_profile_read("decode")
        c2, ms2 = A.attn_profile_read("decode_merge")
        us = (ms1 + ms2) / max(c1, 1) * 1e3
        nbytes = 2 * B * h * m * d * 2 + 2 * B * h * n * d * 2 + 4 * B * h * n
        pairs = B * h * sum(m - n + i + 1 for i in range(n))
        out[name] = {"us": round(us, 1), "merge_us": round(ms2 / max(c2, 1) * 1e3, 1),
                     "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                     "tflops": round(4.0 * d * pairs / (us * 1e-6) / 1e12, 2)}
        del sets, ws, o, lse
        torch.cuda.empty_cache()
    if A.attn_get_device_status() != A.ATTN_OK:
        raise RuntimeError("device watchdog fired in the decoding sweep")
    return out


def run_proj_sweep(args, local):
    """Throughput of the multi-head projections (tensor-bound GEMMs): the QKV
    projection (fused for self-attention) and the output projection, FLOPs
    2 * tokens * d_model * (columns), bytes = operands read once + results; and
    their backward (input and weight gradients: twice the FLOPs; all launches of
    a call, the split reduction included). Rank 0, N=1 only."""
    import torch
    import transformer_scaled_dot_attn_gb300 as A
    from seeded_inputs import PROJ_WORKLOADS
    dev = torch.device("cuda", local)
    peaks, _ = load_peaks()
    out = {}
    for name, (B, n, m, dm, h, d) in PROJ_WORKLOADS.items():
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        hd = h * d
        xq = torch.randn(B, n, dm, device=dev, generator=g).bfloat16()
        xkv = xq if n == m and "self" in name else torch.randn(B, m, dm, device=dev, generator=g).bfloat16()
        w = (torch.randn(dm, 3 * hd, device=dev, generator=g) / dm ** 0.5).bfloat16()
        wo = (torch.randn(hd, dm, device=dev, generator=g) / hd ** 0.5).bfloat16()
        q = torch.empty(B, h, n, d, dtype=torch.bfloat16, device=dev)
        k = torch.empty(B, h, m, d, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        y = torch.empty(B, n, dm, dtype=torch.bfloat16, device=dev)
        gq = torch.randn(B, h, n, d, device=dev, generator=g).bfloat16()
        gk = torch.randn(B, h, m, d, device=dev, generator=g).bfloat16()
        gv = torch.randn(B, h, m, d, device=dev, generator=g).bfloat16()
        gy = torch.randn(B, n, dm, device=dev, generator=g).bfloat16()
        dxq = torch.empty(B, n, dm, dtype=torch.bfloat16, device=dev)
        dxkv = dxq if xkv is xq else torch.empty(B, m, dm, dtype=torch.bfloat16, device=dev)
        dw = torch.empty(dm, 3 * hd, dtype=torch.bfloat16, device=dev)
        d_o = torch.empty(B, h, n, d, dtype=torch.bfloat16, device=dev)
        dwo = torch.empty(hd, dm, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(A.attn_qkv_projection_bwd_workspace_bytes(B, n, m, dm, h, d),
                             A.attn_out_projection_bwd_workspace_bytes(B, n, dm, h, d), 16),
                         dtype=torch.uint8, device=dev)
        res = {}
        for kind in ("qkv", "out", "qkv_bwd", "out_bwd"):
            def call():
                if kind == "qkv":
                    A.attn_qkv_projection(xq, xkv, w, h, d, q=q, k=k, v=v)
                elif kind == "out":
                    A.attn_out_projection(q, wo, y=y)
                elif kind == "qkv_bwd":
                    A.attn_qkv_projection_bwd(xq, xkv, w, gq, gk, gv, dx_q=dxq, dx_kv=dxkv, dw_qkv=dw,
                                              workspace=ws)
                else:
                    A.attn_out_projection_bwd(q, wo, gy, d_o=d_o, dw_o=dwo, workspace=ws)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            A.attn_profile_enable(True)
            A.attn_profile_read("proj")
            iters = 30
            for _ in range(iters):
                call()
            torch.cuda.synchronize()
            A.attn_profile_enable(False)
            c, ms = A.attn_profile_read("proj")
            us = ms / iters * 1e3  # a cross-attention QKV projection is two launches per call
            xkv_b = 0 if xkv is xq else B * m * dm
            if kind == "qkv":
                flops = 2.0 * B * n * dm * hd + 2.0 * B * m * dm * 2 * hd
                nbytes = 2 * (B * n * dm + xkv_b + dm * 3 * hd + B * n * hd + 2 * B * m * hd)
            elif kind == "out":
                flops = 2.0 * B * n * hd * dm
                nbytes = 2 * (B * n * hd + hd * dm + B * n * dm)
            elif kind == "qkv_bwd":
                flops = 2 * (2.0 * B * n * dm * hd + 2.0 * B * m * dm * 2 * hd)
                # reads x, W, dQ, dK, dV; writes dx and dW
                nbytes = 2 * (B * n * dm + xkv_b + dm * 3 * hd + B * n * hd + 2 * B * m * hd +
                              B * n * dm + xkv_b + dm * 3 * hd)
            else:
                flops = 2 * 2.0 * B * n * hd * dm
                nbytes = 2 * (B * n * hd + hd * dm + B * n * dm + B * n * hd + hd * dm)
            tf = flops / (us * 1e-6) / 1e12
            res[kind] = {"us": round(us, 1), "launches_per_call": round(c / iters, 2), "tflops": round(tf, 1),
                         "frac_peak": round(tf / peaks["bf16_tflops"], 3),
                         "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
        out[name] = res
        del xq, xkv, w, wo, q, k, v, y, gq, gk, gv, gy, dxq, dxkv, dw, d_o, dwo, ws
        torch.cuda.empty_cache()
    if A.attn_get_device_status() != A.ATTN_OK:
        raise RuntimeError("device watchdog fired in the projection sweep")
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed steps before the warm-up so clocks settle (0 for profiler runs)")
    ap.add_argument("--chunks", type=int, default=0,
                    help="head chunks of the end-to-end host step (0: the library chooses)")
    ap.add_argument("--only", choices=("decode", "proj"),
                    help="run only the decoding or the projection sweep and print it (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.only is not None:
        fn = run_decode_sweep if args.only == "decode" else run_proj_sweep
        print(json.dumps({args.only: fn(args, 0)}), flush=True)
        return
    world, rank, local = dist_setup()
    w = WORKLOADS[args.workload]
    config = workload_config(w, world)

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = []
        sample, threads = "", 0
        seconds = max(1.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
        for st in range(args.warmup + args.steps):
            tf, t, sample, threads = oracle_sample(w, seconds)
            if st >= args.warmup:
                per_step.append((tf, t))
        value = statistics.median(tf for tf, _ in per_step)
        ms = statistics.median(t for _, t in per_step) * 1e3
        sample = f"per step: {sample} (fp64 C oracle)"
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    res = run_gpu(args, w, world, rank, local)
    sweep = decode_sweep = proj_sweep = None
    if world == 1 and not args.no_sweep:
        sweep = run_sweep(args, local)
        decode_sweep = run_decode_sweep(args, local)
        proj_sweep = run_proj_sweep(args, local)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, t, sample, threads = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": round(tf, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
    if rank != 0:
        return
    peak = res["peaks"]["bf16_tflops"]
    line = {
        "metric": METRIC, "value": round(res["value"], 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (i.i.d. N(0,1) bf16, seeded)", "config": config,
        "frac_of_bf16_peak": round(res["value"] / world / peak, 4),
        "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
        "gpu_launches": res["launches"], "clocks": res["clocks"], "kernels": res["kernels"],
    }
    if sweep is not None:
        line["sweep"] = sweep
    if decode_sweep is not None:
        line["decode_sweep"] = decode_sweep
    if proj_sweep is not None:
        line["proj_sweep"] = proj_sweep
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
