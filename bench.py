#!/usr/bin/env python
"""Throughput of the attention forward on GB300, one JSON line on stdout.

A step is one whole forward pass (one fa_fwd call) over one batch of synthetic
[B, H, N, D] inputs.  Default workload: bf16, B=4, H=16, N=4096, D=128, non-causal,
scale 1/sqrt(128) -- the shape the pages analyse, and the workload the throughput
metric is quoted on.  Metric: attention TFLOPS = 4*B*H*N^2*D / t (halved when causal).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs under torchrun: every rank is an independent replica on its own GPU (the
forward has no exchange step), per-GPU work is fixed ("scaling": "weak"), and value
is the total work of all ranks over the max-over-ranks time.

Timing: W untimed warm-up steps, then exactly K steps between a barrier +
cudaDeviceSynchronize on both sides, timed with CUDA events on the launching stream.
Consecutive steps alternate between two input sets of 192 MiB each (together larger
than the 129 MB L2), so no step starts with its inputs resident in L2.
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

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
_CSRC = os.path.join(ROOT, "attention_forward_04_gb300", "csrc")
# sources whose change invalidates a stored traffic capture
KERNEL_SRCS = {"fwd": [os.path.join(_CSRC, f) for f in ("fa_tc.cu", "tc_common.cuh", "ptx.cuh")],
               "fwd256": [os.path.join(_CSRC, f) for f in ("fa_tc256.cu", "tc_common.cuh", "ptx.cuh")],
               "simt": [os.path.join(_CSRC, "fa_simt.cu")],
               "bwd": [os.path.join(_CSRC, f) for f in ("fa_bwd.cu", "bwd_common.cuh", "tc_common.cuh",
                                                         "ptx.cuh")],
               "bwd256": [os.path.join(_CSRC, f) for f in ("fa_bwd256.cu", "bwd_common.cuh",
                                                            "tc_common.cuh", "ptx.cuh")]}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(op: str = "fwd") -> str:
    """sha256[:16] of the kernel sources' code: comments and whitespace are left out, so an
    edit to a comment does not retire a traffic capture of unchanged code."""
    import re
    h = hashlib.sha256()
    for path in KERNEL_SRCS[op]:
        with open(path, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                  # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(key: str, op: str = "fwd"):
    """dram read+write bytes per launch (per call for the backward) from an ncu capture, if
    it matches the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(key)
    if not e or e.get("kernel_sha256_16") != kernel_hash(op):
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons for one GPU."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [s for (t, s) in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
            window = "around-timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            for name, val in zip(names, s[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][2]), "reasons": sorted(reasons),
                "power_w_max": max((num(s[3]) or 0.0) for s in inside),
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------ CPU oracle leg
def time_oracle(w, budget_s: float, host_qkv, threads: int = 0):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload: whole
    (b, h) slices, as many as fit the time budget (at least one), on `threads` host
    threads (0: all cores).  Returns (tflops, seconds, slices, threads)."""
    import numpy as np
    import oracle
    BH = w.B * w.H
    q, k, v = (t.reshape(1, BH, w.N, w.D) for t in host_qkv)
    threads = threads or oracle.default_threads()
    # estimate the cost of one slice from a probe of 64 rows spread over the slice
    rows = np.unique(np.linspace(0, w.N - 1, min(w.N, 64)).astype(np.int64))
    q0, k0, v0 = (t[:, :1].double().numpy() for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.attention_rows(q0, k0, v0, w.scale, w.causal, np.zeros_like(rows), rows, threads)
    per_row = (time.perf_counter() - t0) / len(rows)
    per_slice = per_row * w.N
    ns = int(max(1, min(BH, budget_s // max(per_slice, 1e-9))))
    qs, ks, vs = (t[:, :ns].double().numpy() for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.attention_fwd(qs, ks, vs, w.scale, w.causal, threads)
    dt = time.perf_counter() - t0
    flops = w.flops * ns / BH
    return flops / dt / 1e12, dt, ns, threads


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from attention_forward_04_gb300.inputs import make_qkv
    oracle.build()
    q, k, v = make_qkv(w.with_(B=1, H=1))
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    threads = oracle.default_threads()
    # size each step so the whole run ends within about two minutes
    probe = np.arange(min(w.N, 16), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention_rows(q64, k64, v64, w.scale, w.causal, np.zeros_like(probe), probe, threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    per_step_budget = min(2.0, 120.0 / max(1, args.steps + args.warmup))
    nrows = int(max(1, min(w.N, per_step_budget / max(per_row, 1e-9))))
    rng = np.random.default_rng(0)
    flops = 0.0
    elapsed = 0.0
    for step in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(w.N, size=nrows, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, w.scale, w.causal, np.zeros_like(rows), rows, threads)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            elapsed += dt
            keys = (rows + 1) if w.causal else np.full_like(rows, w.N)
            flops += float(np.sum(4.0 * keys * w.D))
    value = flops / elapsed / 1e12
    sample = ("%d random query rows of one (b, h) slice per step (of %d rows x %d slices), "
              "fp64 three-pass oracle, %d threads" % (nrows, w.N, w.B * w.H, threads))
    line = {"impl": "reference", "metric": "attention fwd TFLOPS (4*B*H*N^2*D/t)", "value": value,
            "unit": "TFLOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args.gpus, input_set_bytes(w)),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_e2e_pipelined(torch, dev, steps, host_in, dev_in, host_out, dev_out, compute):
    """End-to-end steps through the public API, pipelined the way a caller streaming batches
    would: step i's host->device copies (one stream per input tensor, so several copy
    engines share the link), its call, and its device->host copies (one more stream) overlap
    the neighbouring steps' stages.  Two device buffer sets alternate; events keep every
    buffer's writer after its previous reader.  Every step still copies all its inputs in
    and all its results out.  Returns the elapsed milliseconds."""
    s_in = [torch.cuda.Stream(dev) for _ in host_in]
    s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [[torch.cuda.Event() for _ in host_in] for _ in range(2)]
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("cmp", "out")}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(s_cmp)
    for s_ in s_in:
        s_.wait_event(start)
    s_out.wait_event(start)
    for i in range(steps):
        b = i & 1
        for x, (d, h) in enumerate(zip(dev_in[b], host_in)):
            if i >= 2:
                s_in[x].wait_event(ev["cmp"][b])   # the call of step i-2 has read buffer set b
            with torch.cuda.stream(s_in[x]):
                d.copy_(h, non_blocking=True)
            ev_in[b][x].record(s_in[x])
            s_cmp.wait_event(ev_in[b][x])
        if i >= 2:
            s_cmp.wait_event(ev["out"][b])         # step i-2's results have been copied out
        compute(b, s_cmp)
        ev["cmp"][b].record(s_cmp)
        s_out.wait_event(ev["cmp"][b])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out, dev_out[b]):
                h.copy_(d, non_blocking=True)
        ev["out"][b].record(s_out)
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def aggregate_over_ranks(ms_local: float, units_local: float, steps: int, world: int,
                         all_reduce_max=None):
    """Whole-job throughput of independent replicas: every rank timed its own `steps` steps
    (ms_local); the job time is the slowest rank's, and the value is the units all ranks
    processed (units_local per step per rank) over that time, in units per second.
    all_reduce_max(x) returns the max of x over ranks (None for a single process)."""
    ms = ms_local if all_reduce_max is None or world == 1 else float(all_reduce_max(ms_local))
    return ms, units_local * steps * world / (ms / 1e3)


def torch_all_reduce_max(device):
    import torch
    import torch.distributed as dist

    def f(x):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return f


L2_BYTES = 129 * 10**6          # GB300 L2
FLUSH_BYTES = 256 * 2**20


def l2_note(set_bytes):
    if set_bytes > L2_BYTES:
        return ("two alternating input sets of %.0f MiB each (> 129 MB L2); no flush"
                % (set_bytes / 2**20))
    return ("input sets of %.2f MiB (< 129 MB L2): L2 flushed before every timed call (a "
            "256 MiB buffer written between calls, outside the per-call CUDA event pairs)"
            % (set_bytes / 2**20))


def flush_buffer(torch, dev, set_bytes):
    """A buffer larger than L2 to write between timed calls, when one input set fits in L2."""
    if set_bytes > L2_BYTES:
        return None
    return torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)


def timed_calls(torch, stream, step, steps, flush):
    """Device milliseconds of step(0) .. step(steps - 1) on `stream` (the current stream).
    Without a flush buffer the two alternating input sets evict each other from L2 and one
    event pair brackets the back-to-back calls.  With one, the buffer is written before every
    call and each call has its own event pair, so the writes stay outside the timed spans."""
    def event():
        return torch.cuda.Event(enable_timing=True)
    if flush is None:
        ev0, ev1 = event(), event()
        ev0.record(stream)
        for i in range(steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)
    pairs = [(event(), event()) for _ in range(steps)]
    for i, (a, b) in enumerate(pairs):
        flush.fill_(i & 0x7F)
        a.record(stream)
        step(i)
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs)


def input_set_bytes(w, op="fwd"):
    """Bytes of one input set of a step: Q, K, V (forward); Q, K, V, O, dO and LSE (backward)."""
    n = w.B * w.H * w.N * w.D
    es = {"fp32": 4, "fp8": 1}.get(w.dtype, 2)
    return 3 * n * es if op == "fwd" else 5 * n * es + 4 * w.B * w.H * w.N


def config_of(w, gpus, set_bytes):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
            "dtype": w.dtype, "scale": w.scale, "qk_mult": w.qk_mult,
            "layout": "[B,H,N,D] contiguous", "parallelism": "replicas x%d" % gpus,
            "l2": l2_note(set_bytes)}


# ------------------------------------------------------------------ backward
BWD_METRIC = "attention bwd TFLOPS (10*B*H*N^2*D/t)"


def bwd_flops(w) -> float:
    """Algorithmic backward FLOPs: five N x N x D products per slice (S, dP, dV, dQ, dK),
    2*N^2*D each, halved for the causal mask.  The kernels recompute S and dP once more
    (seven products); that extra work is not counted."""
    return 2.5 * w.flops


def bwd_launches_per_call(w) -> int:
    """Kernels one fa_bwd call launches: dQ (which forms delta) and dK/dV (fp32 on the CUDA
    cores, and 16-bit at D <= 128), or dQ, dV and dK (16-bit at D = 256)."""
    return 3 if w.D == 256 and w.dtype != "fp32" else 2


def time_oracle_bwd(w, budget_s: float, host):
    """The fp64 backward oracle, as it stands, on whole (b, h) slices within the budget."""
    from oracle.backward import attention_bwd
    q, k, v, do = (t.reshape(1, w.B * w.H, w.N, w.D) for t in host)
    args = [t[:, :1].double().numpy() for t in (q, k, v, do)]
    t0 = time.perf_counter()
    attention_bwd(*args, w.scale, w.causal)
    per_slice = time.perf_counter() - t0
    ns = int(max(1, min(w.B * w.H, budget_s // max(per_slice, 1e-9))))
    args = [t[:, :ns].double().numpy() for t in (q, k, v, do)]
    t0 = time.perf_counter()
    attention_bwd(*args, w.scale, w.causal)
    dt = time.perf_counter() - t0
    return bwd_flops(w) * ns / (w.B * w.H) / dt / 1e12, dt, ns


def run_reference_bwd(args, w):
    """The backward oracle timed as the reference arm: whole slices, bounded per step."""
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    from oracle.backward import attention_bwd
    from attention_forward_04_gb300.inputs import make_dout, make_qkv
    one = w.with_(B=1, H=1)
    args64 = [t.double().numpy() for t in (*make_qkv(one), make_dout(one))]
    elapsed = 0.0
    steps = 0
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        attention_bwd(*args64, w.scale, w.causal)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            elapsed += dt
            steps += 1
        if elapsed > 120.0:
            break
    value = bwd_flops(w) / (w.B * w.H) * steps / elapsed / 1e12
    sample = "one whole (b, h) slice per step (of %d), fp64 numpy backward oracle" % (w.B * w.H)
    line = {"impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": elapsed / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(config_of(w, args.gpus, input_set_bytes(w, "bwd")), op="bwd"),
            "cpu_baseline": {"value": value, "unit": "TFLOPS",
                             "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_bwd(args, w):
    """Backward pass: a step is one fa_bwd call (dQ-with-delta and dK/dV kernels) over resident
    Q, K, V, O, LSE, dO; the forward that produces O and LSE runs before timing."""
    rank, local_rank, world = dist_env()
    import torch
    import torch.distributed as dist
    from attention_forward_04_gb300 import binding, build
    from attention_forward_04_gb300.inputs import TORCH_DTYPES, make_dout, make_qkv

    if rank == 0:
        build.build()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist.barrier()
    else:
        torch.cuda.set_device(0)
    lib = binding.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    code = {"fp32": binding.FA_FP32, "bf16": binding.FA_BF16, "fp16": binding.FA_FP16}[w.dtype]
    B, H, N, D = w.B, w.H, w.N, w.D
    sets = []
    for s in range(2):
        q, k, v = (t.to(dev) for t in make_qkv(w, seed_offset=100 * s + 10 * rank))
        do = make_dout(w, seed_offset=100 * s + 10 * rank).to(dev)
        o, lse = binding.fwd(q, k, v, scale=w.scale, causal=w.causal)
        sets.append((q, k, v, o, lse, do))
    grads = [torch.empty((B, H, N, D), dtype=TORCH_DTYPES[w.dtype], device=dev) for _ in range(3)]
    set_bytes = input_set_bytes(w, "bwd")
    wsb = binding.bwd_workspace_bytes(B, H, N)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def step(i):
        q, k, v, o, lse, do = sets[i & 1]
        st = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                        lse.data_ptr(), grads[0].data_ptr(), grads[1].data_ptr(),
                        grads[2].data_ptr(), ws.data_ptr(), wsb, B, H, N, D, w.scale,
                        int(w.causal), code, sh)
        if st != 0:
            raise binding.FaError(st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, detail = binding.check_device_status()
    if st != 0:
        raise RuntimeError("kernel watchdog after warm-up: %d %s" % (st, detail))
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    flush = flush_buffer(torch, dev, set_bytes)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    ms_local = timed_calls(torch, stream, step, args.steps, flush)
    t_wall1 = time.monotonic()
    if world > 1:
        dist.barrier()
    time.sleep(0.15)
    sampler.stop()
    st, detail = binding.check_device_status()
    if st != 0:
        raise RuntimeError("kernel watchdog in timed region: %d %s" % (st, detail))
    flops_step = bwd_flops(w)
    reduce_max = torch_all_reduce_max(dev) if world > 1 else None
    ms, per_s = aggregate_over_ranks(ms_local, flops_step, args.steps, world, reduce_max)
    per_call_ms = ms_local / args.steps

    # ---- end to end: pinned host Q, K, V, O, LSE, dO -> device -> fa_bwd -> host dQ, dK, dV
    host = [t.cpu().pin_memory() for t in sets[0]]
    hgrads = [torch.empty((B, H, N, D), dtype=TORCH_DTYPES[w.dtype]).pin_memory()
              for _ in range(3)]
    dev_in = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
    dev_out = [[torch.empty_like(g) for g in grads] for _ in range(2)]
    wss = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in range(2)]

    def e2e_call(b, s):
        q, k, v, o, lse, do = dev_in[b]
        binding.bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, dq=dev_out[b][0],
                    dk=dev_out[b][1], dv=dev_out[b][2], workspace=wss[b], stream=s)

    run_e2e_pipelined(torch, dev, 2, host, dev_in, hgrads, dev_out, e2e_call)   # warm-up
    if world > 1:
        dist.barrier()
    e2e_elapsed = run_e2e_pipelined(torch, dev, args.e2e_steps, host, dev_in, hgrads, dev_out,
                                    e2e_call)
    e2e_ms, e2e_per_s = aggregate_over_ranks(e2e_elapsed, flops_step, args.e2e_steps, world,
                                             reduce_max)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in hgrads)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops_step / (per_call_ms / 1e3) / 1e12
    # executed products: S and dP are formed twice (dQ kernel, dK/dV kernel), 14 N^2 D per
    # slice; at D = 256 S^T three times (dQ, dV and dK kernels), 16 N^2 D
    d256 = w.D == 256
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak,
            "traffic": load_traffic("bwd:" + w.name, "bwd256" if d256 else "bwd"),
            "kernel": ("whole fa_bwd call (dQ kernel, which also forms delta, dV kernel and dK "
                       "kernel)" if d256 else "whole fa_bwd call (dQ kernel, which also forms "
                       "delta, and dK/dV kernel)") + "; per-kernel shares in the ncu launch list",
            "peak_source": "%s bf16 dense burst" % peak_src,
            "executed_tflops": (4.0 if d256 else 3.5) * w.flops / (per_call_ms / 1e3) / 1e12}
    if w.dtype == "fp32":
        # the CUDA-core backward: fp32 FFMA peak, SMs x 128 fp32 lanes x 2 FLOP x max SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        roof.update({"bound": "alu", "peak": alu_peak, "frac": achieved / alu_peak,
                     "traffic": None, "kernel": "whole fa_bwd call (the two CUDA-core kernels)",
                     "peak_source": "derived: %d SMs x 128 fp32 lanes x 2 FLOP x max SM clock"
                                    % sms})
    cpu = None
    if args.cpu_budget > 0:
        try:
            tfl, secs, ns = time_oracle_bwd(w, args.cpu_budget, [t.cpu() for t in
                                                                 (sets[0][0], sets[0][1],
                                                                  sets[0][2], sets[0][5])])
            cpu = {"value": tfl, "unit": "TFLOPS", "cores": len(os.sched_getaffinity(0)),
                   "kind": "oracle",
                   "sample": "%d of %d (b,h) slices of %s, whole slices, fp64 numpy backward "
                             "oracle, %.1f s (cores: numpy's BLAS threads)" % (ns, B * H, w.name,
                                                                               secs)}
        except Exception as ex:
            cpu = {"value": None, "unit": "TFLOPS", "cores": None, "kind": "oracle",
                   "sample": "failed: %s" % ex}
    line = {
        "metric": BWD_METRIC, "value": per_s / 1e12, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded torch.randn, cast to %s)" % w.dtype,
        "config": dict(config_of(w, world, set_bytes), op="bwd"),
        "e2e": {"value": e2e_per_s / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "ms_per_step": e2e_ms / args.e2e_steps,
                "pipelining": "host->device copies (one stream per input), the call and "
                              "device->host copies of consecutive steps overlap (two device "
                              "buffer sets)"},
        "gpu_launches": bwd_launches_per_call(w) * args.steps,
        "roofline": roof, "cpu_baseline": cpu,
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ main GPU leg
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle timing (0 skips the CPU leg)")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back calls for the sustained block (0 skips it)")
    ap.add_argument("--op", default="fwd", choices=["fwd", "bwd"],
                    help="fwd: the forward pass (default); bwd: the backward pass (fa_bwd)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from attention_forward_04_gb300.inputs import HEADLINE, WORKLOADS
    w = WORKLOADS[args.workload or HEADLINE]
    if args.op == "bwd":
        if args.impl == "reference":
            return run_reference_bwd(args, w)
        return run_bwd(args, w)
    if args.impl == "reference":
        return run_reference(args, w)

    rank, local_rank, world = dist_env()
    import torch
    import torch.distributed as dist
    from attention_forward_04_gb300 import binding, build
    from attention_forward_04_gb300.inputs import TORCH_DTYPES, make_qkv, make_qkv_fp8

    if rank == 0:
        build.build()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist.barrier()
    else:
        torch.cuda.set_device(0)
    binding.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    fp8 = w.dtype == "fp8"
    code = {"fp32": binding.FA_FP32, "bf16": binding.FA_BF16, "fp16": binding.FA_FP16,
            "fp8": -1}[w.dtype]
    B, H, N, D = w.B, w.H, w.N, w.D
    lib = binding.load_library()

    def inputs(seed_offset):
        # fp8: e4m3 tensors and their per-tensor dequantisation factors
        if fp8:
            return make_qkv_fp8(w, seed_offset=seed_offset)
        return make_qkv(w, seed_offset=seed_offset), (1.0, 1.0, 1.0)

    sets, descales = [], None
    for s in range(2):
        (q, k, v), descales = inputs(100 * s + 10 * rank)
        sets.append(tuple(t.to(dev) for t in (q, k, v)))
    host_set, host_descales = inputs(10 * rank)
    set_bytes = input_set_bytes(w)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16 if fp8 else TORCH_DTYPES[w.dtype],
                    device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def step(i):
        q, k, v = sets[i & 1]
        if fp8:
            st = lib.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, H, N, D, w.scale, int(w.causal), descales[0],
                                descales[1], descales[2], sh)
        else:
            st = binding.fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, D, w.scale, int(w.causal), code, sh)
        if st != 0:
            raise binding.FaError(st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, detail = binding.check_device_status()
    if st != 0:
        raise RuntimeError("kernel watchdog after warm-up: %d %s" % (st, detail))

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)

    flush = flush_buffer(torch, dev, set_bytes)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    ms_local = timed_calls(torch, stream, step, args.steps, flush)
    t_wall1 = time.monotonic()
    if world > 1:
        dist.barrier()
    st, detail = binding.check_device_status()
    if st != 0:
        raise RuntimeError("kernel watchdog in timed region: %d %s" % (st, detail))

    flops_step = w.flops
    reduce_max = torch_all_reduce_max(dev) if world > 1 else None
    ms, per_s = aggregate_over_ranks(ms_local, flops_step, args.steps, world, reduce_max)
    value = per_s / 1e12
    per_launch_ms = ms_local / args.steps

    # ---- sustained: seconds of back-to-back calls on the same inputs, with the clock samples
    # that fall inside them (the K-step region above can be too short for the power cap to act)
    sustained = None
    if args.sustain_s > 0:
        n_sus = max(args.steps, int(args.sustain_s * 1e3 / max(per_launch_ms, 1e-3)) + 1)
        # small inputs are flushed from L2 before every call: bound the host-side work
        n_sus = min(n_sus, 2000 if flush is not None else 200000)
        time.sleep(0.25)
        torch.cuda.synchronize()
        t_sus0 = time.monotonic()
        ms_sus = timed_calls(torch, stream, step, n_sus, flush)
        t_sus1 = time.monotonic()
        st, detail = binding.check_device_status()
        if st != 0:
            raise RuntimeError("kernel watchdog in sustained region: %d %s" % (st, detail))
        sustained = {"steps": n_sus, "ms_per_step": ms_sus / n_sus,
                     "value": flops_step / (ms_sus / n_sus / 1e3) / 1e12, "unit": "TFLOPS",
                     "wall_s": t_sus1 - t_sus0}
    time.sleep(0.15)
    sampler.stop()

    # ---- end to end through the public API: pinned host inputs -> device -> fa.fwd -> host
    hq, hk, hv = (t.pin_memory() for t in host_set)
    ho = torch.empty((B, H, N, D), dtype=o.dtype).pin_memory()
    hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    dev_in = [[torch.empty_like(t, device=dev) for t in host_set] for _ in range(2)]
    dev_out = [[torch.empty_like(o), torch.empty_like(lse)] for _ in range(2)]

    def e2e_call(b, s):
        q_, k_, v_ = dev_in[b]
        if fp8:
            binding.fwd_fp8(q_, k_, v_, *host_descales, scale=w.scale, causal=w.causal,
                            out=dev_out[b][0], lse=dev_out[b][1], stream=s)
        else:
            binding.fwd(q_, k_, v_, scale=w.scale, causal=w.causal, out=dev_out[b][0],
                        lse=dev_out[b][1], stream=s)

    run_e2e_pipelined(torch, dev, 2, (hq, hk, hv), dev_in, (ho, hl), dev_out, e2e_call)  # warm-up
    if world > 1:
        dist.barrier()
    e2e_elapsed = run_e2e_pipelined(torch, dev, args.e2e_steps, (hq, hk, hv), dev_in, (ho, hl),
                                    dev_out, e2e_call)
    e2e_ms, e2e_per_s = aggregate_over_ranks(e2e_elapsed, flops_step, args.e2e_steps, world,
                                             reduce_max)
    e2e_value = e2e_per_s / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops_step / (per_launch_ms / 1e3) / 1e12
    traffic = load_traffic(w.name, "simt" if w.dtype == "fp32" else "fwd256" if w.D == 256 else "fwd")
    if w.dtype == "fp32":
        # fp32 FFMA peak: SMs x 128 fp32 lanes x 2 FLOP x max SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": traffic,
                "peak_source": "derived: %d SMs x 128 fp32 lanes x 2 FLOP x max SM clock" % sms}
    else:
        # e4m3 products run at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense), so
        # their peak is the measured bf16 peak times 2
        ratio = 2.0 if fp8 else 1.0
        src = ("%s bf16 dense burst (MEASURED_PEAKS.json)" % peak_src
               if peak_src == "measured" else "fallback 1.9 PFLOP/s")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak * ratio, "unit": "TFLOP/s",
                "frac": achieved / (peak * ratio), "traffic": traffic,
                "peak_source": src + (" x 2 (e4m3 : bf16 nominal dense ratio)" if fp8 else ""),
                "frac_of_sustained": achieved / (ratio * float(peaks.get("bf16_tflops_sustained", 1700.0))),
                "hbm_gbs_algorithmic": (3 * (1 if fp8 else 2) + 2) * B * H * N * D / (per_launch_ms / 1e3) / 1e9}

    cpu = None
    if args.cpu_budget > 0:
        try:
            tfl, secs, ns, threads = time_oracle(w, args.cpu_budget, host_set)
            cpu = {"value": tfl, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                   "sample": "%d of %d (b,h) slices of %s (N=%d, D=%d, causal=%s), whole "
                             "slices, fp64 three-pass oracle, %.1f s"
                             % (ns, B * H, w.name, N, D, w.causal, secs)}
            # the same oracle on one host thread, on a sample of its own budget
            tfl1, secs1, ns1, _ = time_oracle(w, args.cpu_budget / 2, host_set, threads=1)
            cpu["single_thread"] = {"value": tfl1, "unit": "TFLOPS", "cores": 1,
                                    "sample": "%d of %d (b,h) slices, whole slices, %.1f s"
                                              % (ns1, B * H, secs1)}
        except Exception as ex:  # the CPU leg must not hide the GPU number
            cpu = {"value": None, "unit": "TFLOPS", "cores": None, "kind": "oracle",
                   "sample": "failed: %s" % ex}

    clocks = sampler.summary(t_wall0, t_wall1)
    if sustained is not None:
        sc = sampler.summary(t_sus0, t_sus1)
        sustained["clocks"] = sc
        sus_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        if w.dtype != "fp32":
            ratio = 2.0 if fp8 else 1.0
            sustained["frac_of_sustained_peak"] = sustained["value"] / (ratio * sus_peak)
            sustained["sustained_peak_source"] = (
                "%s bf16 dense sustained (MEASURED_PEAKS.json)%s"
                % (peak_src, " x 2 (e4m3 : bf16 nominal dense ratio)" if fp8 else ""))
            if sc.get("sm_mhz"):
                # tensor rate per SM and clock: 8192 dense bf16/fp16 FLOP (128x128x16 product
                # in 64 cycles, measured with a back-to-back tcgen05.mma microbenchmark), twice
                # that for e4m3
                sms = torch.cuda.get_device_properties(dev).multi_processor_count
                clk_peak = sms * 8192 * ratio * sc["sm_mhz"] * 1e6 / 1e12
                sustained["clock_normalised_peak"] = clk_peak
                sustained["frac_of_clock_normalised_peak"] = sustained["value"] / clk_peak
    line = {
        "metric": "attention fwd TFLOPS (4*B*H*N^2*D/t)",
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else w.dtype,
        "data": ("synthetic (seeded torch.randn, per-tensor e4m3 quantisation; O bf16)" if fp8
                 else "synthetic (seeded torch.randn, cast to %s)" % w.dtype),
        "config": config_of(w, world, set_bytes),
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "ms_per_step": e2e_ms / args.e2e_steps,
                "pipelining": "host->device copies (one stream per input), the call and "
                              "device->host copies of consecutive steps overlap (two device "
                              "buffer sets)"},
        "gpu_launches": args.steps,
        "timing": "value: the K timed steps back to back (a burst); sustained: the same "
                  "calls for --sustain-s seconds",
        "sustained": sustained,
        "roofline": roof,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "pct_of_peak": 100.0 * roof["frac"] if w.dtype != "fp32" else None,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
