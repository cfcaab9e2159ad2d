"""Benchmark of the B300 kernelized linear-attention library.

One JSON line on rank 0.  A step is one causal forward (la_forward_ex: phi,
intra-chunk scores, readout, state carry, state export) over the long
workload B=1, H=16, N=65536, D=Dv=128, bf16, elu+1; ``value`` is tokens/s
(B*N positions, all H heads) with inputs resident in HBM.  The same run
times the batched decode (la_step, B=64, H=16, 4096 tokens from that
forward's final state) and reports it under ``decode``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--decode-steps T] [--no-cpu-baseline]

Multi-GPU runs (torchrun, one process per GPU) are independent replicas:
every rank runs the same workload; value = all ranks' tokens / max time.
``--impl reference`` times the oracle (fp64 CPU loop) on host cores, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "causal linear-attention tokens/sec at 1 B300 and % of roofline; decode steps/sec"
L2_BYTES = 126 * 1024 * 1024
HOST_COVER_CYCLES = 600_000   # ~0.3 ms at 2 GHz
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def alg_bytes(w: wl.Workload) -> int:
    """Algorithmic HBM bytes of one forward: read q, k, v, write out."""
    e = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (2 * w.D + 2 * w.Dv) * e


def alg_flops(w: wl.Workload) -> int:
    """Algorithmic FLOPs of the RNN form per token-head: S update and readout
    (4 Dphi Dv), z update and denominator (3 Dphi), divide (Dv); PRF adds
    the projection and its exponent arguments (4 m D + 2 D + 2 m)."""
    P = w.phi_dim
    f = 4 * P * w.Dv + 3 * P + w.Dv
    if w.feature == "prf":
        f += 4 * w.m * w.D + 2 * w.D + 2 * w.m
    return w.token_heads * f


def alg_bytes_backward(w: wl.Workload) -> int:
    """Algorithmic HBM bytes of one backward: read q, k, v, dout; write dq, dk, dv."""
    e = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (4 * w.D + 3 * w.Dv) * e


def alg_flops_backward(w: wl.Workload) -> int:
    """Algorithmic FLOPs of the backward's RNN form per token-head: the forward
    recomputed (4 P Dv), d phi(q) (2 P Dv), the reverse memory (2 P Dv), d phi(k)
    and dv (4 P Dv), vector terms (10 P + 4 Dv); PRF adds the projections of
    q and k and their chain rule (16 m D)."""
    P = w.phi_dim
    f = 12 * P * w.Dv + 10 * P + 4 * w.Dv
    if w.feature == "prf":
        f += 16 * w.m * w.D
    return w.token_heads * f


def alg_bytes_prefix(w: wl.Workload) -> int:
    """Prefix attention: read k, v and write out per token-head, plus q per head."""
    e = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (w.D + 2 * w.Dv) * e + w.B * w.H * w.D * e


def alg_flops_prefix(w: wl.Workload) -> int:
    """Per token-head: the score (2 D), the state update and readout (4 Dv + 6)."""
    return w.token_heads * (2 * w.D + 4 * w.Dv + 6)


def alg_bytes_rpe(w: wl.Workload) -> int:
    """Kernelized attention with RPE: read q, k, v and b, write out."""
    e = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (2 * w.D + 2 * w.Dv) * e + w.H * (2 * w.N - 1) * 4


def alg_flops_rpe(w: wl.Workload) -> int:
    """The weighted form's work: per (query, key) pair the score (2 Dphi), the
    weight (1) and the accumulation of the value and the denominator
    (2 Dv + 2); N(N+1)/2 pairs per head when causal, N^2 otherwise."""
    pairs = w.N * (w.N + 1) // 2 if w.causal else w.N * w.N
    return w.B * w.H * pairs * (2 * w.phi_dim + 2 * w.Dv + 3)


def decode_bytes_per_step(BH, P, Dv, D, e=2) -> int:
    """S and z read+write (fp32), q, k, v read and out written (dtype)."""
    return BH * (2 * P * Dv * 4 + 2 * P * 4 + (2 * D + 2 * Dv) * e)


# the translation unit of the kernels whose DRAM traffic profiles/traffic.json
# records: the counters stay valid while these files are unchanged
KERNEL_SOURCES = ("common.cuh", "kernels.h", "tc_causal.cu", "tc_ptx.cuh")


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_linear_attention_map_b300", "csrc")
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_workload: str):
    """DRAM bytes per launch from the committed ncu summary, if its source
    digest matches the library as built now; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel_workload)
    except Exception:
        return None
    if not d or d.get("source_digest") != source_digest():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, int(parts[2]), int(parts[3]), parts[4:]))
            except Exception:
                continue
        os.unlink(self.path)
        inwin = [r for r in rows if any(a - 0.06 <= r[0] <= b + 0.06 for a, b in self.windows)]
        window = "timed"
        if not inwin:
            inwin, window = rows, "whole run"
        if not inwin:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inwin:
            for n, v in zip(names, r[3][2:6]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inwin),
                "sm_max_mhz": max(r[2] for r in inwin), "reasons": sorted(reasons),
                "samples": len(inwin), "window": window}


# ------------------------------------------------------------------ our arm

def dist_setup():
    """One process per GPU (torchrun env).  Ranks use NCCL on GPUs; without a
    GPU (host-side tests of the multi-rank logic) they use gloo."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    gpu = torch.cuda.is_available()
    if gpu:
        torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist

        if gpu:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x: float, ws: int) -> float:
    """The slowest rank's time (every rank gets it)."""
    if ws == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step: float, steps: int, ws: int, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (replicas: every rank does the same work)."""
    return units_per_rank_step * steps * ws / (max_ms / 1e3)


def oracle_sample(w: wl.Workload, budget_s: float, cores: int):
    """Heads x positions of the workload that one oracle call covers within
    about ``budget_s``: at least min(B*H, cores) heads, so that every OpenMP
    thread (one head each) has work; positions, then heads, grow by 4x."""
    BH = w.B * w.H
    n_heads = min(BH, max(1, cores))
    n_pos = min(w.N, 1024)
    # cost model from the oracle's loop: ~(4 Dphi Dv + elementwise) per token-head
    per = 4.0 * w.phi_dim * w.Dv + (4 * w.m * w.D if w.feature == "prf" else 0) + 8 * w.D
    rate = 0.5e9 * min(n_heads, cores)   # fp64 flop/s, a rough guess refined by timing
    while n_pos < w.N and n_heads * n_pos * 4 * per / rate <= budget_s:
        n_pos = min(w.N, n_pos * 4)
    while n_pos == w.N and n_heads < BH and min(BH, n_heads * 4) * n_pos * per / rate <= budget_s:
        n_heads = min(BH, n_heads * 4)
    return n_heads, n_pos


def cpu_baseline(w: wl.Workload, q, k, v, W, budget_s=12.0, reps_min=1):
    """The oracle, as it stands, timed on the host cores over a bounded sample
    of the workload (a whole number of calls, each over the same sample)."""
    import oracle

    lib = oracle.load()
    cores = oracle.num_threads(lib)
    BH = w.B * w.H
    Wn = W.double().numpy() if W is not None else None
    n_heads, n_pos = oracle_sample(w, budget_s / 2, cores)

    def part(t, d):
        return t.reshape(BH, w.N, d)[:n_heads, :n_pos].double().numpy()[None]

    qs, ks, vs = part(q, w.D), part(k, w.D), part(v, w.Dv)
    times = []
    while len(times) < reps_min or (sum(times) < budget_s / 2 and len(times) < 50):
        t0 = time.perf_counter()
        oracle.forward(qs, ks, vs, causal=w.causal, feature=w.feature, W=Wn, lib=lib)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    token_heads = n_heads * n_pos
    whole = n_heads == BH and n_pos == w.N
    return {"value": token_heads / w.H / dt, "unit": "tokens/s",
            "cores": min(cores, n_heads), "kind": "oracle",
            "sample": f"{'the whole workload' if whole else 'a sample'}: {n_heads} of {BH} heads x "
                      f"first {n_pos} of {w.N} positions ({token_heads} token-heads), fp64 "
                      f"recurrence, OpenMP over heads ({min(cores, n_heads)} threads of {cores}); "
                      f"median of {len(times)} calls, {dt:.3f} s each; "
                      f"tokens/s = token-heads / H / seconds",
            "seconds_per_call": dt, "calls": len(times), "whole_workload": whole}


def timed_steps(la, fn, args, dev, stream, ws, rank, scrub):
    """W warm-up calls of fn, then K timed ones with CUDA events on ``stream``.
    With ``scrub`` (inputs that fit in L2) every step is timed alone after
    writing the scrub buffer, behind a device-side delay that covers the host
    enqueue; else the K steps are timed back to back.  Returns (total ms, the
    slowest rank's; library launches in the timed region; clocks)."""
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
    for _ in range(args.warmup):
        fn()
        if scrub is not None:
            scrub.fill_(1.0)
    barrier(ws)
    n0 = la.la_launch_count()
    t_wall0 = time.time()
    if scrub is not None:
        total_ms = 0.0
        for _ in range(args.steps):
            scrub.fill_(1.0)
            # a device-side delay before the start event, so that the host has
            # queued the whole call by the time the GPU reaches it (the timed
            # region then holds only the call's device work; host cost per
            # call is in e2e)
            torch.cuda._sleep(HOST_COVER_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            total_ms += e0.elapsed_time(e1)
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        e1.synchronize()
        total_ms = e0.elapsed_time(e1)
    barrier(ws)
    sampler.mark(t_wall0, time.time())
    # stop polling nvidia-smi once the timed region is over: its driver queries
    # would otherwise slow the host-bound e2e steps of the small workloads
    clocks = sampler.stop() if rank == 0 else None
    launches = la.la_launch_count() - n0
    return max_over_ranks(total_ms, ws), launches, clocks


def hbm_roofline(ab, af, seconds, kernel):
    """The roofline entry for ``ab`` algorithmic bytes and ``af`` flops done in
    ``seconds``: the slower of the HBM time and the dense bf16 tensor time."""
    pk, pk_kind = peaks()
    t_hbm = ab / (pk["hbm_gbs"] * 1e9)
    t_flop = af / (pk["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_flop else "tensor"
    if bound == "hbm":
        achieved, peak, unit = ab / seconds / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = af / seconds / 1e12, pk["bf16_tflops"], "TFLOP/s"
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4),
            "peak_source": f"{pk_kind} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})",
            "kernel": kernel, "alg_bytes_per_launch": ab, "alg_flops_per_launch": af,
            "roofline_time_us": round(max(t_hbm, t_flop) * 1e6, 2),
            "frac_of_roofline_time": round(max(t_hbm, t_flop) / seconds, 4)}


def measure_forward(la, w: wl.Workload, args, dev, stream, ws, rank, with_e2e=True,
                    with_cpu=True, keep_state=False):
    """Time la_forward_ex over workload ``w`` (inputs resident in HBM), then
    the same metric end to end through la_forward_host; returns the entry
    for the JSON line (and the exported state when ``keep_state``)."""
    q, k, v = wl.make_qkv(w)
    W = wl.make_W(w.m, w.D) if w.feature == "prf" else None
    dq, dk, dv = (t.to(dev) for t in (q, k, v))
    fm = la.FeatureMap("prf", W.to(dev)) if W is not None else None
    out = torch.empty((w.B, w.H, w.N, w.Dv), dtype=dq.dtype, device=dev)
    P = w.phi_dim
    S_out = torch.empty((w.B, w.H, P, w.Dv), dtype=torch.float32, device=dev)
    z_out = torch.empty((w.B, w.H, P), dtype=torch.float32, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (dq, dk, dv))
    flush = in_bytes + out.numel() * out.element_size() < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def fwd():
        la.la_forward_ex(dq, dk, dv, causal=w.causal, feature_map=fm, out=out, S_out=S_out,
                         z_out=z_out, stream=stream)

    total_ms, launches, clocks = timed_steps(la, fwd, args, dev, stream, ws, rank, scrub)
    ms_step = total_ms / args.steps
    tokens = w.B * w.N
    value = job_rate(tokens, args.steps, ws, total_ms)

    pk, pk_kind = peaks()
    fwd_s = ms_step / 1e3
    ab, af = alg_bytes(w), alg_flops(w)
    t_hbm = ab / (pk["hbm_gbs"] * 1e9)
    t_flop = af / (pk["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_flop else "tensor"
    if bound == "hbm":
        achieved, peak, unit = ab / fwd_s / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = af / fwd_s / 1e12, pk["bf16_tflops"], "TFLOP/s"
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(w.name),
                "peak_source": f"{pk_kind} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})",
                "kernel": "la_forward_ex (all of its launches, timed together)",
                "alg_bytes_per_launch": ab, "alg_flops_per_launch": af,
                "roofline_time_us": round(max(t_hbm, t_flop) * 1e6, 2),
                "frac_of_roofline_time": round(max(t_hbm, t_flop) / fwd_s, 4)}
    entry = {"workload": w.name, "value": value, "unit": "tokens/s", "ms_per_step": ms_step,
             "steps": args.steps, "warmup": args.warmup,
             "dtype": "bf16" if w.dtype == "bf16" else "f32",
             "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "Dv": w.Dv,
                        "causal": w.causal, "feature": w.feature, "m": w.m,
                        "token_heads_per_step": w.token_heads,
                        "l2": "L2 flushed between steps (host enqueue hidden behind a device "
                              "delay before the start event)" if flush else
                        f"inputs ({in_bytes / 1e6:.0f} MB) larger than L2"},
             "roofline": roofline, "gpu_launches": launches,
             # the same rate counted per (position, head): tokens/s x H
             "token_heads_per_s": value * w.H}
    if clocks:
        entry["clocks"] = clocks

    if with_e2e:
        # end to end through the C ABI with host buffers: la_forward_host copies
        # q, k, v in and out back, overlapping both copy directions with the
        # forward by head groups
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def e2e_step():
            la.la_forward_host(hq, hk, hv, causal=w.causal, feature_map=fm, out=hout,
                               stream=stream)

        for _ in range(2):
            e2e_step()
        barrier(ws)
        e_steps = max(3, min(args.steps, 10))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
        entry["e2e"] = {"value": job_rate(tokens, e_steps, ws, e_ms), "unit": "tokens/s",
                        "h2d_bytes_per_step": in_bytes,
                        "d2h_bytes_per_step": out.numel() * out.element_size(), "steps": e_steps,
                        "path": "la_forward_host (C ABI): pinned host q, k, v in, out back; "
                                "copies in both directions overlapped with the forward by "
                                "head groups"}
        del hq, hk, hv, hout

    if with_cpu and rank == 0 and ws == 1:
        log(f"timing the oracle on host cores ({w.name}) ...")
        entry["cpu_baseline"] = cpu_baseline(w, q, k, v, W, budget_s=args.cpu_budget)
    del dq, dk, dv, out, scrub
    if keep_state:
        return entry, S_out, z_out
    del S_out, z_out
    return entry


def oracle_timed(w: wl.Workload, call, budget_s: float, cost_factor: float, what: str):
    """Time ``call(n_heads, n_pos)`` (an oracle routine over the first heads and
    positions of the workload) on a bounded sample; the sample is sized like
    oracle_sample with its cost scaled by ``cost_factor``."""
    import oracle

    cores = oracle.num_threads(oracle.load())
    n_heads, n_pos = oracle_sample(w, budget_s / 2 / cost_factor, cores)
    times = []
    while not times or (sum(times) < budget_s / 2 and len(times) < 20):
        t0 = time.perf_counter()
        call(n_heads, n_pos)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    th = n_heads * n_pos
    BH = w.B * w.H
    return {"value": th / w.H / dt, "unit": "tokens/s", "cores": min(cores, n_heads), "kind": "oracle",
            "sample": f"{n_heads} of {BH} heads x first {n_pos} of {w.N} positions ({th} token-heads), "
                      f"fp64 {what}, OpenMP over heads; median of {len(times)} calls, {dt:.3f} s each"}


def backward_path(w: wl.Workload) -> str:
    """Which kernels la_backward runs for workload ``w`` (the library's rule)."""
    if w.dtype == "bf16" and w.feature == "elu1" and w.D == w.Dv and w.D in (64, 128):
        return ("tensor cores (tcgen05 kind::f16): fp16 operands, dnum as an fp16 hi + lo pair, "
                "per-chunk power-of-two scales, fp32 accumulation")
    return "CUDA cores, fp32 arithmetic"


def measure_backward(la, w: wl.Workload, args, dev, stream, ws, rank, with_cpu=True):
    """la_backward over workload ``w`` (inputs resident in HBM)."""
    q, k, v = wl.make_qkv(w)
    do = wl.make_dout(w)
    W = wl.make_W(w.m, w.D) if w.feature == "prf" else None
    dq_, dk_, dv_, ddo = (t.to(dev) for t in (q, k, v, do))
    fm = la.FeatureMap("prf", W.to(dev)) if W is not None else None
    gq, gk, gv = torch.empty_like(dq_), torch.empty_like(dk_), torch.empty_like(dv_)
    nbytes = sum(t.numel() * t.element_size() for t in (dq_, dk_, dv_, ddo, gq, gk, gv))
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if nbytes < 2 * L2_BYTES else None

    def fn():
        la.la_backward(dq_, dk_, dv_, ddo, causal=w.causal, feature_map=fm, dq=gq, dk=gk, dv=gv, stream=stream)

    total_ms, launches, clocks = timed_steps(la, fn, args, dev, stream, ws, rank, scrub)
    ms = total_ms / args.steps
    entry = {"workload": w.name, "value": job_rate(w.B * w.N, args.steps, ws, total_ms), "unit": "tokens/s",
             "ms_per_step": ms, "gpu_launches": launches,
             "roofline": hbm_roofline(alg_bytes_backward(w), alg_flops_backward(w), ms / 1e3,
                                      "la_backward (all of its launches, timed together)"),
             "l2": "L2 flushed between steps" if scrub is not None else "tensors larger than L2",
             "path": backward_path(w)}
    if clocks:
        entry["clocks"] = clocks
    if with_cpu and rank == 0 and ws == 1:
        import oracle

        BH = w.B * w.H
        Wn = W.double().numpy() if W is not None else None

        def call(nh, npos):
            sl = lambda t, c: t.reshape(BH, w.N, c)[:nh, :npos].double().numpy()[None]
            oracle.backward(sl(q, w.D), sl(k, w.D), sl(v, w.Dv), sl(do, w.Dv), causal=w.causal,
                            feature=w.feature, W=Wn)

        log(f"timing the backward oracle ({w.name}) ...")
        entry["cpu_baseline"] = oracle_timed(w, call, args.cpu_budget / 2, 3.0, "reverse-mode recurrence")
    del dq_, dk_, dv_, ddo, gq, gk, gv, scrub
    return entry


def measure_rpe(la, w: wl.Workload, args, dev, stream, ws, rank, with_cpu=True):
    """la_forward_rpe over the workload with its relative-position log-weights."""
    q, k, v = wl.make_qkv(w)
    b = wl.make_rpe_bias(w)
    dq_, dk_, dv_, db = (t.to(dev) for t in (q, k, v, b))
    out = torch.empty_like(dv_)
    nbytes = sum(t.numel() * t.element_size() for t in (dq_, dk_, dv_, out))
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if nbytes < 2 * L2_BYTES else None

    def fn():
        la.la_forward_rpe(dq_, dk_, dv_, db, causal=w.causal, out=out, stream=stream)

    total_ms, launches, clocks = timed_steps(la, fn, args, dev, stream, ws, rank, scrub)
    ms = total_ms / args.steps
    entry = {"workload": w.name, "value": job_rate(w.B * w.N, args.steps, ws, total_ms), "unit": "tokens/s",
             "ms_per_step": ms, "gpu_launches": launches,
             "roofline": hbm_roofline(alg_bytes_rpe(w), alg_flops_rpe(w), ms / 1e3,
                                      "rpe_tc_kernel (one launch; chunk-against-chunk weighted form)"),
             "l2": "L2 flushed between steps" if scrub is not None else "tensors larger than L2"}
    if clocks:
        entry["clocks"] = clocks
    if with_cpu and rank == 0 and ws == 1:
        import oracle

        BH = w.B * w.H

        def call(nh, npos):
            sl = lambda t, c: t.reshape(BH, w.N, c)[:nh, :npos].double().numpy()[None]
            bb = np64_bias(b, nh, npos, w)
            oracle.rpe(sl(q, w.D), sl(k, w.D), sl(v, w.Dv), bb, causal=w.causal)

        log(f"timing the RPE oracle ({w.name}) ...")
        entry["cpu_baseline"] = oracle_timed(w, call, args.cpu_budget / 2, w.N / 64.0,
                                             "quadratic weighted form")
    del dq_, dk_, dv_, db, out, scrub
    return entry


def np64_bias(b, nh, npos, w):
    """The log-weight rows of the first nh heads (head index bh % H) for the
    first npos positions: b[h, t + N - 1] for |t| < npos."""
    rows = [int(i % w.H) for i in range(nh)]
    c = w.N - 1
    return b[rows][:, c - (npos - 1):c + npos].double().numpy()


def measure_prefix(la, w: wl.Workload, args, dev, stream, ws, rank, with_cpu=True):
    """la_prefix_attention over the workload's keys and values with its query token."""
    q = wl.make_prefix_q(w)
    _, k, v = wl.make_qkv(w)
    dq_, dk_, dv_ = (t.to(dev) for t in (q, k, v))
    out = torch.empty_like(dv_)
    nbytes = sum(t.numel() * t.element_size() for t in (dk_, dv_, out))
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if nbytes < 2 * L2_BYTES else None

    def fn():
        la.la_prefix_attention(dq_, dk_, dv_, out=out, stream=stream)

    total_ms, launches, clocks = timed_steps(la, fn, args, dev, stream, ws, rank, scrub)
    ms = total_ms / args.steps
    entry = {"workload": w.name, "value": job_rate(w.B * w.N, args.steps, ws, total_ms), "unit": "tokens/s",
             "ms_per_step": ms, "gpu_launches": launches,
             "roofline": hbm_roofline(alg_bytes_prefix(w), alg_flops_prefix(w), ms / 1e3,
                                      "prefix_attn_kernel (one launch)"),
             "l2": "L2 flushed between steps" if scrub is not None else "tensors larger than L2"}
    if clocks:
        entry["clocks"] = clocks
    if with_cpu and rank == 0 and ws == 1:
        import oracle

        BH = w.B * w.H

        def call(nh, npos):
            oracle.prefix_attention(q.reshape(BH, w.D)[:nh].double().numpy()[None],
                                    k.reshape(BH, w.N, w.D)[:nh, :npos].double().numpy()[None],
                                    v.reshape(BH, w.N, w.Dv)[:nh, :npos].double().numpy()[None])

        log(f"timing the prefix-attention oracle ({w.name}) ...")
        entry["cpu_baseline"] = oracle_timed(w, call, args.cpu_budget / 2, 1.0 / max(1, w.D // 8),
                                             "RNN cell over the prefix")
    del dq_, dk_, dv_, out, scrub
    return entry


def run_ours(args):
    ws, rank, local = dist_setup()
    import causal_linear_attention_map_b300 as la
    from causal_linear_attention_map_b300 import build as _build

    if rank == 0:
        _build.build()
    barrier(ws)
    la.load()
    w = workload_of(args)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    head, S_out, z_out = measure_forward(la, w, args, dev, stream, ws, rank,
                                         with_cpu=not args.no_cpu_baseline, keep_state=True)
    result = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": ws,
              "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": head["dtype"], "data": "synthetic (seeded N(0,1)/sqrt(D))",
              "config": dict(head["config"],
                             parallelism="replicas" if ws > 1 else "single GPU"),
              "roofline": head["roofline"], "e2e": head.get("e2e"),
              "gpu_launches": head["gpu_launches"], "token_heads_per_s": head["token_heads_per_s"]}
    if "cpu_baseline" in head:
        result["cpu_baseline"] = head["cpu_baseline"]
    if head.get("clocks"):
        result["clocks"] = head["clocks"]

    if args.decode_steps > 0 and w.causal and w.D == wl.DECODE_D and w.feature == "elu1":
        result["decode"] = run_decode(la, args, S_out, z_out, dev, stream, ws)
    del S_out, z_out

    # every other workload of the method's table, measured the same way in the
    # same process (each with its own clocks, roofline and oracle baseline)
    if args.all_configs and args.seq_len == 0 and args.workload == wl.LONG_65536.name:
        configs = {w.name: {k_: v_ for k_, v_ in head.items() if k_ != "config"}}
        for other in wl.WORKLOADS.values():
            if other.name == w.name:
                continue
            log(f"measuring {other.name} ...")
            configs[other.name] = measure_forward(la, other, args, dev, stream, ws, rank,
                                                  with_cpu=not args.no_cpu_baseline)
            torch.cuda.empty_cache()
        result["configs"] = configs
        result["gpu_launches"] = sum(c["gpu_launches"] for c in configs.values()) + \
            result.get("decode", {}).get("launches", 0)
    if args.extras and args.seq_len == 0 and args.workload == wl.LONG_65536.name:
        # the gradients over every workload, and softmax attention as an RNN
        # over the long and image workloads' keys and values
        result["backward"] = {}
        for other in wl.WORKLOADS.values():
            log(f"measuring the backward of {other.name} ...")
            result["backward"][other.name] = measure_backward(la, other, args, dev, stream, ws, rank,
                                                              with_cpu=not args.no_cpu_baseline)
            torch.cuda.empty_cache()
        result["prefix_attention"] = {}
        for other in (wl.LONG_65536, wl.IMAGE_3072):
            log(f"measuring prefix attention over {other.name} ...")
            result["prefix_attention"][other.name] = measure_prefix(la, other, args, dev, stream, ws, rank,
                                                                    with_cpu=not args.no_cpu_baseline)
            torch.cuda.empty_cache()
        # kernelized attention with a Toeplitz relative-position weight, over the
        # non-causal and the image workloads
        result["rpe"] = {}
        for other in (wl.NONCAUSAL_4096, wl.IMAGE_3072):
            log(f"measuring attention with RPE over {other.name} ...")
            result["rpe"][other.name] = measure_rpe(la, other, args, dev, stream, ws, rank,
                                                    with_cpu=not args.no_cpu_baseline)
            torch.cuda.empty_cache()
        result["gpu_launches"] += sum(e["gpu_launches"] for e in result["backward"].values()) + \
            sum(e["gpu_launches"] for e in result["prefix_attention"].values()) + \
            sum(e["gpu_launches"] for e in result["rpe"].values())
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def l2_copy_gbs(dev, stream, nbytes: int) -> float:
    """Read+write GB/s of a device copy of ``nbytes`` into another buffer,
    both small enough to stay in L2 together; best of 5 timed loops."""
    nbytes = min(nbytes, L2_BYTES // 3)
    a = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    b = torch.empty_like(a)
    for _ in range(10):
        b.copy_(a)
    best = 0.0
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(50):
            b.copy_(a)
        e1.record(stream)
        e1.synchronize()
        best = max(best, 2 * a.numel() * 4 * 50 / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del a, b
    return best


def run_decode(la, args, S_fwd, z_fwd, dev, stream, ws):
    """4096 batched decode steps from the forward's final state replicated
    into B=64 rows (same 16 heads in every row)."""
    B, H, D = wl.DECODE_B, wl.DECODE_H, wl.DECODE_D
    T = args.decode_steps
    S0 = S_fwd[0:1].expand(B, -1, -1, -1).contiguous()
    z0 = z_fwd[0:1].expand(B, -1, -1).contiguous()
    log(f"generating {T} decode steps of inputs ...")
    qs = torch.empty((T, B, H, D), dtype=torch.bfloat16, device=dev)
    ks = torch.empty_like(qs)
    vs = torch.empty_like(qs)
    for t in range(T):
        a, b, c = wl.make_decode_qkv(t)
        qs[t].copy_(a, non_blocking=True); ks[t].copy_(b, non_blocking=True)
        vs[t].copy_(c, non_blocking=True)
    out = torch.empty((T, B, H, D), dtype=torch.bfloat16, device=dev)
    S = S0.clone()
    z = z0.clone()

    def run(nsteps):
        for t in range(nsteps):
            la.la_step(S, z, qs[t], ks[t], vs[t], out=out[t], stream=stream)

    run(min(T, 32))
    S.copy_(S0); z.copy_(z0)
    barrier(ws)
    n0 = la.la_launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(T)
    e1.record(stream)
    e1.synchronize()
    launches = la.la_launch_count() - n0
    ms = max_over_ranks(e0.elapsed_time(e1), ws)
    # the same steps replayed from a CUDA graph (chunks of 64 launches)
    G = 64
    graph_ms = None
    if T % G == 0:
        S.copy_(S0); z.copy_(z0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(dev)
        base = torch.zeros(1, dtype=torch.int64)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(g, stream=gs):
                for t in range(G):
                    la.la_step(S, z, qs[t], ks[t], vs[t], out=out[t], stream=gs)
        del base
        S.copy_(S0); z.copy_(z0)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(gs)
        with torch.cuda.stream(gs):
            for _ in range(T // G):
                g.replay()
        e1.record(gs)
        e1.synchronize()
        graph_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    pk, pk_kind = peaks()
    bps = decode_bytes_per_step(B * H, D, D, D)
    ach = bps * T / (ms / 1e3) / 1e9
    l2 = l2_copy_gbs(dev, stream, S.numel() * 4)
    res = {"steps_per_s": job_rate(T, 1, ws, ms), "tokens_per_s": job_rate(T * B, 1, ws, ms),
           "ms_total": ms, "us_per_step": ms * 1e3 / T, "decode_steps": T, "B": B, "H": H,
           "D": D, "launches": launches,
           "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                        "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                        "alg_bytes_per_step": bps, "peak_source": pk_kind,
                        "note": "the 64 MB fp32 state fits in L2 (126 MB), so steps may run "
                                "from L2; frac can exceed 1"},
           # the same bytes against an L2-resident copy of the state's size, measured here
           "roofline_l2": {"bound": "l2", "achieved": round(ach, 1), "peak": round(l2, 1),
                           "unit": "GB/s", "frac": round(ach / l2, 4),
                           "peak_source": "measured in this run: device copy of a buffer of the "
                                          "state's size into another (read + write bytes), "
                                          "both resident in L2, best of 5 x 50 copies"}}
    if graph_ms is not None:
        res["graph"] = {"steps_per_s": job_rate(T, 1, ws, graph_ms), "ms_total": graph_ms,
                        "launches_per_graph": G,
                        "note": "steps replayed with the state reset; same 4096 inputs"}
    return res


def workload_of(args) -> wl.Workload:
    w = wl.WORKLOADS[args.workload]
    if args.seq_len > 0 and args.seq_len != w.N:
        name = w.name.replace(f"_N{w.N}_", f"_N{args.seq_len}_")
        w = w.with_(N=args.seq_len, name=name)
    return w


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores.  One step
    is one oracle call over the same bounded sample of the workload (the
    whole workload when it fits the per-step budget); every step is timed."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    w = workload_of(args)
    q, k, v = wl.make_qkv(w)
    W = wl.make_W(w.m, w.D) if w.feature == "prf" else None
    lib = oracle.load()
    cores = oracle.num_threads(lib)
    budget = 60.0 / max(1, args.steps + args.warmup)
    n_heads, n_pos = oracle_sample(w, budget, cores)
    BH = w.B * w.H
    Wn = W.double().numpy() if W is not None else None

    def part(t, d):
        return t.reshape(BH, w.N, d)[:n_heads, :n_pos].double().numpy()[None]

    qs, ks, vs = part(q, w.D), part(k, w.D), part(v, w.Dv)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(qs, ks, vs, causal=w.causal, feature=w.feature, W=Wn, lib=lib)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    token_heads = n_heads * n_pos
    value = token_heads / w.H / dt
    whole = n_heads == BH and n_pos == w.N
    threads = min(cores, n_heads)
    sample = (f"{'the whole workload' if whole else 'a sample'}: {n_heads} of {BH} heads x first "
              f"{n_pos} of {w.N} positions ({token_heads} token-heads) per step, fp64 recurrence, "
              f"OpenMP over heads ({threads} threads of {cores}); median of {len(times)} timed "
              f"steps; tokens/s = token-heads / H / seconds")
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1)/sqrt(D))", "impl": "reference",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "Dv": w.Dv,
                   "causal": w.causal, "feature": w.feature, "m": w.m,
                   "step": "one oracle call over " + ("the whole workload" if whole else
                                                      f"{token_heads} token-heads of it")},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=wl.LONG_65536.name, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=wl.DECODE_STEPS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle time per workload for cpu_baseline")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the backward and prefix-attention measurements")
    ap.add_argument("--no-all-configs", dest="all_configs", action="store_false",
                    help="measure only the named workload (default: the long workload plus "
                         "every other workload of the table under 'configs')")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run the named workload at this N instead (a smaller case for profiler "
                         "captures; the JSON line then names the shortened workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
