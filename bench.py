"""Benchmark: exact attention forward (bf16) on GB300, one JSON line.

A step is one fa_fwd call over the whole workload (B=1, Hq=Hkv=16,
Lq=Lk=16384, D=128, non-causal by default): every stage of the forward
(tile schedule, TMA loads, S = QK^T, masking, online softmax, P.V, epilogue)
runs inside it.  The metric is matrix TFLOP/s, 4*B*Hq*Lq*Lk*D per step
(halved when causal).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

With N > 1 (torchrun, one rank per GPU) every rank runs its own copy of the
workload (the problem partitions over batch and heads with no exchange), and
`value` is the total work of all ranks over the slowest rank's time.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (BF16) and fraction of GB300 dense BF16 peak"
FALLBACK_BF16_TFLOPS = 1900.0
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


L2_MIB = 126  # L2 of one GB300 as the runtime reports it
NOMINAL_BF16_TFLOPS = 2250.0  # dense BF16 tensor peak of one GB300, nominal


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--full-oracle", action="store_true",
                    help="reference arm: time the oracle over the whole workload (every output row) per step")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of the extra back-to-back pass reported as 'sustained' (0 = none)")
    return ap.parse_args(argv)


def workload_config(w, world: int) -> dict:
    """The `config` object of a bench line; both arms print the same one."""
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lq": w.Lq, "Lk": w.Lk, "D": w.D, "Dv": w.Dv,
            "causal": w.causal, "flops_per_step": w.flops(),
            "parallelism": f"replicas{world}" if world > 1 else "single"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


FALLBACK_HBM_GBS = 6800.0


def decode_rows(R):
    """Query rows the tensor-core decode kernel's softmax carries for R packed rows."""
    return 4 if R <= 4 else 8 if R <= 8 else 16


def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


KERNEL_SOURCES = ("exact_attention_07_gb300/csrc/fa_fwd_kernel.cuh", "exact_attention_07_gb300/csrc/ptx_sm103.cuh",
                  "exact_attention_07_gb300/csrc/fa_params.h")
BWD_SOURCES = ("exact_attention_07_gb300/csrc/fa_bwd.cu", "exact_attention_07_gb300/csrc/ptx_sm103.cuh",
               "exact_attention_07_gb300/csrc/fa_bwd.h")
DECODE_SOURCES = ("exact_attention_07_gb300/csrc/fa_decode_tc.cu", "exact_attention_07_gb300/csrc/fa_decode.cu",
                  "exact_attention_07_gb300/csrc/ptx_sm103.cuh", "exact_attention_07_gb300/csrc/fa_decode.h")


def kernel_source_hash(read=None, sources=KERNEL_SOURCES) -> str:
    """sha256 of the kernel sources with comments and blank space removed, so
    that only code changes invalidate recorded counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sources:
        if read is None:
            with open(os.path.join(ROOT, f)) as fh:
                text = fh.read()
        else:
            text = read(f)
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.strip() for line in text.splitlines() if line.strip())
        h.update(text.encode())
    return h.hexdigest()


def profiled_traffic(workload: str, sources=KERNEL_SOURCES, prefix="fa_fwd"):
    """DRAM bytes per launch (per step for decode) from the committed ncu
    summary of this workload, or None when there is none or the kernel changed
    since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = dict(line.strip().split(": ", 1) for line in text.splitlines()
                  if line.strip().startswith(("traffic_bytes_per_launch:", "kernel_source_sha256:")))
    if fields.get("kernel_source_sha256") != kernel_source_hash(sources=sources):
        return None
    return int(fields["traffic_bytes_per_launch"])


def job_rate(secs: float, units: float, world: int, device=None) -> tuple[float, float]:
    """Whole-job throughput over all ranks: (sum of units) / (max of seconds).

    Every rank passes its own timed seconds and processed units; all ranks get
    (units per second, slowest rank's seconds).  With one rank it is local.
    """
    if world <= 1:
        return (units / secs if secs > 0 else 0.0), secs
    import torch
    import torch.distributed as dist
    t = torch.tensor([secs], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    secs_max, units_all = float(t.item()), float(u.item())
    return (units_all / secs_max if secs_max > 0 else 0.0), secs_max


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    def __init__(self, gpu_index: int, path: str | None = None):
        self.gpu = gpu_index
        self.path = path
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
            if self.path:
                with open(self.path, "w") as f:
                    f.write(SMI_FIELDS + "\n" + "\n".join(self.lines) + "\n")

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle timing

def cpu_oracle_rate(w, inputs, seconds: float, rng_seed: int = 0, full: bool = False):
    """Time the fp64 oracle on sampled output rows for about `seconds` (or,
    with `full`, on every output row of the workload).

    Returns (TFLOP/s, threads, description, timed seconds).  FLOPs per row
    follow the metric (4*Lk*D, halved on average when causal).
    """
    import numpy as np

    import oracle
    rng = np.random.default_rng(rng_seed)
    if w.bwd:
        return _cpu_backward_rate(w, inputs, seconds)
    if w.window is not None:
        return _cpu_variant_rate(w, inputs, seconds)
    if full:
        if w.varlen:
            q, k, v, cq, ck = inputs
            t0 = time.perf_counter()
            oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=w.scale, causal=w.causal)
        else:
            q, k, v = inputs
            t0 = time.perf_counter()
            oracle.attention(q, k, v, scale=w.scale, causal=w.causal)
        dt = time.perf_counter() - t0
        return w.flops() / dt / 1e12, oracle.num_cpus(), f"the whole workload, every output row ({dt:.1f} s)", dt
    if w.varlen:
        q, k, v, cq, ck = inputs
        Tq = q.shape[0]
        total_rows = w.Hq * Tq
        per_row = w.flops() / total_rows

        def run(rows):
            oracle.attention_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=w.scale, causal=w.causal, rows=rows)
    else:
        q, k, v = inputs
        total_rows = w.B * w.Hq * w.Lq
        per_row = w.flops() / total_rows

        def run(rows):
            oracle.attention(q, k, v, scale=w.scale, causal=w.causal, rows=rows)
    threads = oracle.num_cpus()
    n = max(threads, 16)
    t0 = time.perf_counter()
    run(rng.integers(0, total_rows, n))
    dt = time.perf_counter() - t0
    n = int(min(total_rows, max(n, n * seconds / max(dt, 1e-6))))
    rows = rng.integers(0, total_rows, n)
    t0 = time.perf_counter()
    run(rows)
    dt = time.perf_counter() - t0
    return per_row * n / dt / 1e12, threads, f"{n} random output rows of {total_rows} ({dt:.1f} s)", dt


def _cpu_backward_rate(w, inputs, seconds: float):
    """Time the fp64 backward oracle on the last n query rows of one head
    (all keys; with bottom-right causal alignment those rows keep the same
    masks as in the full problem).  FLOPs: 10 * D per allowed (query, key)
    pair, the metric's accounting of the five matrix products."""
    import numpy as np

    import oracle
    from oracle.backward import attention_bwd
    from workloads import grad_output
    if w.varlen:
        # the first sequence of the packed batch, as a dense [1, H, L, D] problem
        q, k, v, cq, ck = inputs
        do = grad_output(tuple(q.shape), w.seed)
        q0, q1, k0, k1 = int(cq[0]), int(cq[1]), int(ck[0]), int(ck[1])
        q, do = (t[q0:q1].permute(1, 0, 2)[None] for t in (q, do))
        k, v = (t[k0:k1].permute(1, 0, 2)[None] for t in (k, v))
        Lq, Lk, what = q1 - q0, k1 - k0, "the first sequence, "
    else:
        q, k, v = inputs
        do = grad_output(tuple(q.shape), w.seed)
        Lq, Lk, what = w.Lq, w.Lk, ""

    def run(n):
        sl = slice(Lq - n, Lq)
        t0 = time.perf_counter()
        attention_bwd(q[:1, :1, sl], k[:1, :1], v[:1, :1], do[:1, :1, sl], w.scale, w.causal)
        dt = time.perf_counter() - t0
        rows = np.arange(Lq - n, Lq)
        pairs = np.minimum(rows + 1 + (Lk - Lq), Lk).clip(0).sum() if w.causal else n * Lk
        return dt, 10.0 * w.D * float(pairs)
    n = min(Lq, 64)
    dt, _ = run(n)
    n = int(min(Lq, max(n, n * seconds / max(dt, 1e-6))))
    dt, fl = run(n)
    return (fl / dt / 1e12, oracle.num_cpus(), f"backward of {what}the last {n} query rows of one head ({dt:.1f} s)",
            dt)


def _cpu_variant_rate(w, inputs, seconds: float):
    """Time the fp64 variant oracle on the last n query rows of one head (whole
    1024-row blocks of the oracle); FLOPs: 4 * D per allowed pair."""
    import numpy as np

    import oracle
    from oracle.variants import attention_variant
    q, k, v = inputs

    def run(n):
        rows = np.arange(w.Lq - n, w.Lq)
        t0 = time.perf_counter()
        attention_variant(q[:1, :1], k[:1, :1], v[:1, :1], w.scale, w.window, rows=rows)
        dt = time.perf_counter() - t0
        c = rows + (w.Lk - w.Lq)
        lo = np.maximum(0, c - w.window[0]) if w.window[0] >= 0 else np.zeros_like(c)
        hi = np.minimum(w.Lk - 1, c + w.window[1]) if w.window[1] >= 0 else np.full_like(c, w.Lk - 1)
        return dt, 4.0 * w.D * float(np.maximum(hi - lo + 1, 0).sum())
    n = 1024
    dt, _ = run(n)
    n = int(min(w.Lq, max(1024, (n * seconds / max(dt, 1e-6)) // 1024 * 1024)))
    dt, fl = run(n)
    return fl / dt / 1e12, oracle.num_cpus(), f"last {n} query rows of one head ({dt:.1f} s)", dt


# ------------------------------------------------------------------ reference arm

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from workloads import dense_inputs, varlen_inputs
    inputs = varlen_inputs(w) if w.varlen else dense_inputs(w)
    # Each step times the oracle on a bounded sample of the workload (about
    # 150 s over the whole run), or with --full-oracle on all of it.  The value
    # is the sampled rate; ms_per_step is the time each step actually took.
    budget = 150.0 / max(1, args.steps + args.warmup)
    rates, secs = [], []
    for i in range(args.warmup + args.steps):
        r, threads, desc, dt = cpu_oracle_rate(w, inputs, budget, rng_seed=i, full=args.full_oracle)
        if i >= args.warmup:
            rates.append(r)
            secs.append(dt)
    value = statistics.median(rates)
    ms = statistics.mean(secs) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "sampled": not args.full_oracle,
            "full_step_ms_at_this_rate": w.flops() / (value * 1e12) * 1e3,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def main(argv=None):
    args = parse_args(argv)
    from workloads import HEADLINE, WORKLOADS
    w = WORKLOADS[args.workload or HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    import exact_attention_07_gb300 as fa
    from workloads import dense_inputs, varlen_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    fa.load_library()
    stream = torch.cuda.current_stream(dev)

    # inputs resident in HBM (seeded on the CPU, copied once)
    host_inputs = varlen_inputs(w) if w.varlen else dense_inputs(w)
    if w.varlen and w.bwd:
        from workloads import grad_output
        q, k, v, cq, ck = (t.to(dev) for t in host_inputs)
        maxl = max(w.seqlens)
        do = grad_output(tuple(q.shape), w.seed).to(dev)
        o_f, lse_f = fa.fa_fwd_varlen(q, k, v, cq, ck, maxl, maxl, causal=w.causal)  # computed once
        dk_b = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv_b = torch.empty(k.shape, dtype=torch.float32, device=dev)
        ws_b = torch.empty(fa.bwd_varlen_workspace(len(w.seqlens), q.shape[0], w.Hq), dtype=torch.uint8,
                           device=dev)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):  # o receives dQ
            return fa.fa_bwd_varlen(qq, kk, vv, o_f, lse_f, do, cq, ck, maxl, maxl, causal=w.causal, dq=o,
                                    dk=dk_b, dv=dv_b, workspace=ws_b)
        out_shape, lse_shape = tuple(q.shape), (w.Hq, q.shape[0])
    elif w.varlen:
        q, k, v, cq, ck = (t.to(dev) for t in host_inputs)
        maxl = max(w.seqlens)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):
            return fa.fa_fwd_varlen(qq, kk, vv, cq, ck, maxl, maxl, causal=w.causal, out=o, lse=lse)
        out_shape, lse_shape = tuple(q.shape), (w.Hq, q.shape[0])
    elif w.bwd:
        from workloads import grad_output
        q, k, v = (t.to(dev) for t in host_inputs)
        do = grad_output(tuple(q.shape), w.seed).to(dev)
        if w.window is not None:  # the forward's outputs, computed once
            o_f, lse_f = fa.fa_fwd_variant(q, k, v, window=w.window)
        else:
            o_f, lse_f = fa.fa_fwd(q, k, v, causal=w.causal)
        dk_b = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv_b = torch.empty(k.shape, dtype=torch.float32, device=dev)
        ws_b = torch.empty(fa.bwd_workspace(w.B, w.Hq, w.Lq), dtype=torch.uint8, device=dev)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):  # o receives dQ
            if w.window is not None:
                return fa.fa_bwd_variant(qq, kk, vv, o_f, lse_f, do, window=w.window, dq=o, dk=dk_b, dv=dv_b,
                                         workspace=ws_b)
            return fa.fa_bwd(qq, kk, vv, o_f, lse_f, do, causal=w.causal, dq=o, dk=dk_b, dv=dv_b, workspace=ws_b)
        out_shape, lse_shape = tuple(q.shape), (w.B, w.Hq, w.Lq)
    elif w.fp8:
        from workloads import fp8_signs
        q, k, v = (t.to(dev) for t in host_inputs)
        signs_d = torch.from_numpy(fp8_signs(w.D, w.seed)).float().to(dev)
        prep = fa.fp8_prepare(q, k, v, signs_d)  # inputs prepared once, as a KV cache would be

        def step(o=None, lse=None):
            return fa.fa_fwd_fp8(prep, w.B, w.Hq, w.Hkv, w.Lq, w.Lk, causal=w.causal, out=o, lse=lse)
        out_shape, lse_shape = tuple(q.shape), (w.B, w.Hq, w.Lq)
    elif w.window is not None:
        q, k, v = (t.to(dev) for t in host_inputs)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):
            return fa.fa_fwd_variant(qq, kk, vv, window=w.window, out=o, lse=lse)
        out_shape, lse_shape = tuple(q.shape), (w.B, w.Hq, w.Lq)
    elif w.decode:
        q, k, v = (t.to(dev) for t in host_inputs)
        ws_bytes, n_splits = fa.splitkv_workspace(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):
            return fa.fa_fwd_splitkv(qq, kk, vv, causal=w.causal, out=o, lse=lse, workspace=ws)
        out_shape, lse_shape = tuple(q.shape), (w.B, w.Hq, w.Lq)
    elif w.Dv != w.D:
        q, k, v = (t.to(dev) for t in host_inputs)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):
            return fa.fa_fwd_hdim(qq, kk, vv, causal=w.causal, out=o, lse=lse)
        out_shape, lse_shape = (w.B, w.Hq, w.Lq, w.Dv), (w.B, w.Hq, w.Lq)
    else:
        q, k, v = (t.to(dev) for t in host_inputs)

        def step(o=None, lse=None, qq=q, kk=k, vv=v):
            return fa.fa_fwd(qq, kk, vv, causal=w.causal, out=o, lse=lse)
        out_shape, lse_shape = tuple(q.shape), (w.B, w.Hq, w.Lq)
    o = torch.empty(out_shape, dtype=torch.float32, device=dev)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    if w.bwd:  # Q, K, V, dO, O, LSE in; dQ, dK, dV out
        in_bytes += do.numel() * 2 + o_f.numel() * 4 + dk_b.numel() * 8
        what = "Q+K+V+dO+O+dQ+dK+dV"
    else:
        what = "Q+K+V+O"
    ws_mib = (in_bytes + o.numel() * 4) / 2**20
    # A working set under twice the L2 could be served from it across steps:
    # then every step is timed alone, after a write of a buffer twice the L2
    flush_buf = None
    if ws_mib < 2 * L2_MIB:
        flush_buf = torch.empty(int(2 * L2_MIB) << 20, dtype=torch.uint8, device=dev)
        l2_note = ("operands (%s = %.0f MiB) under 2x the %d MiB L2: L2 flushed by a %d MiB write before each "
                   "step, each step timed by its own events" % (what, ws_mib, L2_MIB, 2 * L2_MIB))
    else:
        l2_note = "operands larger than L2 (%s = %.0f MiB vs %d MiB L2); no flush" % (what, ws_mib, L2_MIB)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        step(o, lse)
    fa.fa_check()
    launches_per_step = fa.fa_last_launch_count()

    # ---- device-resident timed region
    # raw clock samples of the timed region (the JSON line carries their summary)
    out_dir = os.environ.get("FA_BENCH_OUT_DIR", os.path.join(ROOT, "bench_out"))
    os.makedirs(out_dir, exist_ok=True)
    clk_path = os.path.join(out_dir, f"bench_clocks_rank{rank}.csv")
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(dev.index, clk_path) as clocks:
        barrier()
        if flush_buf is None:
            start.record(stream)
            for _ in range(args.steps):
                step(o, lse)
            end.record(stream)
        else:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in evs:
                flush_buf.zero_()
                e0.record(stream)
                step(o, lse)
                e1.record(stream)
        barrier()
    fa.fa_check()
    if flush_buf is None:
        secs = start.elapsed_time(end) / 1e3
    else:
        secs = sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3

    # A shorter second pass with one event pair per step gives the median and
    # the minimum step time next to the whole-loop mean above (which is the
    # reported value).
    n_dist = min(args.steps, 50)
    evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dist)]
    barrier()
    for e0, e1 in evd:
        if flush_buf is not None:
            flush_buf.zero_()
        e0.record(stream)
        step(o, lse)
        e1.record(stream)
    barrier()
    fa.fa_check()
    step_ms = sorted(e0.elapsed_time(e1) for e0, e1 in evd)
    step_stats = {"median": statistics.median(step_ms), "min": step_ms[0], "n": n_dist,
                  "note": "one event pair per step, after the timed loop"}
    flops_step = w.flops()
    rate, secs_max = job_rate(secs, flops_step * args.steps, world, dev)
    value = rate / 1e12
    ms_per_step = secs_max / args.steps * 1e3

    # ---- sustained: one more back-to-back pass of at least --sustained-seconds
    # with its own clock record.  The timed loop above is short and runs at
    # burst clocks; a pass of seconds settles under the power cap.
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = int(min(200000, max(args.steps, math.ceil(args.sustained_seconds / max(secs / args.steps, 1e-7)))))
        sus_secs, done = 0.0, 0
        barrier()
        with ClockSampler(dev.index, os.path.join(out_dir, f"bench_clocks_sustained_rank{rank}.csv")) as sclk:
            barrier()
            while done < n_sus:
                m = n_sus - done if flush_buf is None else min(1000, n_sus - done)
                if flush_buf is None:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(m):
                        step(o, lse)
                    e1.record(stream)
                    e1.synchronize()
                    sus_secs += e0.elapsed_time(e1) / 1e3
                else:  # the L2 flush between steps, as in the timed loop, outside the events
                    evs2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                            for _ in range(m)]
                    for e0, e1 in evs2:
                        flush_buf.zero_()
                        e0.record(stream)
                        step(o, lse)
                        e1.record(stream)
                    evs2[-1][1].synchronize()
                    sus_secs += sum(e0.elapsed_time(e1) for e0, e1 in evs2) / 1e3
                done += m
            barrier()
        fa.fa_check()
        sus_rate, sus_max = job_rate(sus_secs, flops_step * n_sus, world, dev)
        sustained = {"value": sus_rate / 1e12, "unit": "TFLOP/s", "steps": n_sus, "seconds": sus_max,
                     "ms_per_step": sus_max / n_sus * 1e3, "clocks": sclk.summary(),
                     "note": "a second back-to-back pass of at least %.1f s after the timed loop"
                             % args.sustained_seconds}

    # ---- end to end through the public API with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        e2e_in = list(host_inputs)
        if w.bwd:  # the backward's own inputs: Q, K, V (cu_seqlens), dO and the forward's O and LSE
            e2e_in += [do.cpu(), o_f.cpu(), lse_f.cpu()]
        pin = [t.pin_memory() for t in e2e_in]
        h_o = torch.empty(out_shape, dtype=torch.float32).pin_memory()
        h_l = torch.empty(lse_shape, dtype=torch.float32).pin_memory()
        h_extra = []  # dK and dV of the backward
        if w.bwd:
            h_extra = [torch.empty(dk_b.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
        # Two slots of device inputs and outputs, so that a step's copies can
        # overlap the neighbouring steps' kernels: step i's host->device copy runs
        # on one copy stream, its kernels on the compute stream, its
        # device->host read on another copy stream.  Every step still moves all
        # of its inputs and outputs.
        slots = 2
        d_ins = [[torch.empty_like(t, device=dev) for t in pin] for _ in range(slots)]
        if w.bwd:
            d_outs = [(torch.empty_like(o), torch.empty_like(dk_b), torch.empty_like(dv_b)) for _ in range(slots)]
        else:
            d_outs = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(slots)]

        def call(d_in, outs):
            """One step of the public API on device buffers (on the current stream)."""
            if w.bwd:
                dq_o, dk_o, dv_o = outs
            else:
                o_o, l_o = outs
            if w.varlen and w.bwd:  # Q, K, V, cu_q, cu_k, dO, O, LSE
                fa.fa_bwd_varlen(d_in[0], d_in[1], d_in[2], d_in[6], d_in[7], d_in[5], d_in[3], d_in[4], maxl, maxl,
                                 causal=w.causal, dq=dq_o, dk=dk_o, dv=dv_o, workspace=ws_b)
            elif w.varlen:
                fa.fa_fwd_varlen(d_in[0], d_in[1], d_in[2], d_in[3], d_in[4], maxl, maxl, causal=w.causal,
                                 out=o_o, lse=l_o)
            elif w.decode:
                fa.fa_fwd_splitkv(d_in[0], d_in[1], d_in[2], causal=w.causal, out=o_o, lse=l_o, workspace=ws)
            elif w.bwd and w.window is not None:
                fa.fa_bwd_variant(d_in[0], d_in[1], d_in[2], d_in[4], d_in[5], d_in[3], window=w.window, dq=dq_o,
                                  dk=dk_o, dv=dv_o, workspace=ws_b)
            elif w.bwd:
                fa.fa_bwd(d_in[0], d_in[1], d_in[2], d_in[4], d_in[5], d_in[3], causal=w.causal, dq=dq_o, dk=dk_o,
                          dv=dv_o, workspace=ws_b)
            elif w.window is not None:
                fa.fa_fwd_variant(d_in[0], d_in[1], d_in[2], window=w.window, out=o_o, lse=l_o)
            elif w.fp8:  # bf16 inputs from the host, prepared and attended on the device
                fa.fp8_prepare(d_in[0], d_in[1], d_in[2], signs_d, prepared=prep)
                fa.fa_fwd_fp8(prep, w.B, w.Hq, w.Hkv, w.Lq, w.Lk, causal=w.causal, out=o_o, lse=l_o)
            elif w.Dv != w.D:
                fa.fa_fwd_hdim(d_in[0], d_in[1], d_in[2], causal=w.causal, out=o_o, lse=l_o)
            else:
                fa.fa_fwd(d_in[0], d_in[1], d_in[2], causal=w.causal, out=o_o, lse=l_o)

        def read_back(outs):
            h_o.copy_(outs[0], non_blocking=True)
            if w.bwd:
                h_extra[0].copy_(outs[1], non_blocking=True)
                h_extra[1].copy_(outs[2], non_blocking=True)
            else:
                h_l.copy_(outs[1], non_blocking=True)

        def serial_step():
            for d, h in zip(d_ins[0], pin):
                d.copy_(h, non_blocking=True)
            call(d_ins[0], d_outs[0])
            read_back(d_outs[0])

        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(slots)]
        ev_k = [torch.cuda.Event() for _ in range(slots)]
        ev_out = [torch.cuda.Event() for _ in range(slots)]

        def pipelined_step(i):
            sl = i % slots
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_k[sl])  # the kernels two steps back are done with these inputs
                for d, h in zip(d_ins[sl], pin):
                    d.copy_(h, non_blocking=True)
                ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            stream.wait_event(ev_out[sl])  # the read-back two steps back is done with these outputs
            call(d_ins[sl], d_outs[sl])
            ev_k[sl].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[sl])
                read_back(d_outs[sl])
                ev_out[sl].record(s_out)

        def timed(run, n):
            barrier()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for i in range(n):
                run(i)
            for e in ev_out:
                stream.wait_event(e)
            t1.record(stream)
            barrier()
            fa.fa_check()
            return t0.elapsed_time(t1) / 1e3

        for i in range(3):
            serial_step()
        ser_secs = timed(lambda i: serial_step(), args.e2e_steps)
        for i in range(3):
            pipelined_step(i)
        e2e_secs = timed(pipelined_step, args.e2e_steps)
        e2e_rate, e2e_secs = job_rate(e2e_secs, flops_step * args.e2e_steps, world, dev)
        ser_rate, ser_secs = job_rate(ser_secs, flops_step * args.e2e_steps, world, dev)
        h2d = sum(t.numel() * t.element_size() for t in pin)
        d2h = h_o.numel() * 4 + (sum(t.numel() * 4 for t in h_extra) if w.bwd else h_l.numel() * 4)
        e2e = {"value": e2e_rate / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_secs / args.e2e_steps * 1e3,
               "pipelined": "2 slots: step i's host->device copy and step i-1's read-back overlap other steps' "
                            "kernels on their own streams",
               "serial": {"value": ser_rate / 1e12, "ms_per_step": ser_secs / args.e2e_steps * 1e3,
                          "note": "copy in, compute, read back, one step at a time on one stream"}}

    # ---- roofline of the attention kernel (the only kernel of a dense step)
    peak, peak_sus, peak_kind = measured_peaks()
    if w.decode:
        # HBM-bound: the least bytes of a step over the whole step's time
        # (partial kernel + merge), so the partial kernel alone runs faster
        # than this figure says
        hbm, hbm_kind = measured_hbm()
        achieved = w.hbm_bytes() / (secs / args.steps) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": profiled_traffic(w.name, DECODE_SOURCES, "fa_decode"),
                    "peak_kind": f"{hbm_kind} HBM copy",
                    "algorithmic_bytes_per_step": w.hbm_bytes(), "splits": n_splits,
                    "kernel": ("fa_decode_tc_kernel<%d,%d>" % (w.D, decode_rows(w.Hq // w.Hkv * w.Lq))
                               if w.Hq // w.Hkv * w.Lq >= 2
                               else "fa_decode_partial_kernel<%d,*>" % w.D) + " + fa_decode_merge_kernel<%d>" % w.D,
                    "timed": "whole step (both launches)"}
    elif w.fp8:
        # e4m3 tensor-core peak: the measured bf16 GEMM peak times the nominal
        # fp8/bf16 ratio (4.5 / 2.25 dense PFLOP/s)
        achieved = flops_step / (secs / args.steps) / 1e12
        peak8 = peak * 2.0
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak8, "unit": "TFLOP/s",
                    "frac": achieved / peak8, "traffic": profiled_traffic(w.name),
                    "peak_kind": f"{peak_kind} burst bf16 GEMM x 2 (nominal e4m3/bf16 ratio)",
                    "frac_of_bf16_peak": achieved / peak,
                    "kernel": "fa_fwd_sm103_kernel<128,%s,false,4>" % str(w.causal).lower()}
    elif w.bwd:
        # both launches of the step (preprocess + gradient kernel) over the step's time
        achieved = flops_step / (secs / args.steps) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": profiled_traffic(w.name, BWD_SOURCES, "fa_bwd"),
                    "peak_kind": f"{peak_kind} burst bf16 GEMM", "frac_of_sustained": achieved / peak_sus,
                    "kernel": ("fa_varlen_schedule_kernel + fa_bwd_pre_varlen_kernel<%d> + fa_bwd_sm103_kernel<%s,true>"
                               if w.varlen else "fa_bwd_pre_kernel<%d> + fa_bwd_sm103_kernel<%s,false>")
                              % (w.D, str(w.causal).lower()),
                    "timed": "whole step (all launches)"}
    else:
        achieved = flops_step / (secs / args.steps) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                    "peak_kind": f"{peak_kind} burst bf16 GEMM", "frac_of_sustained": achieved / peak_sus,
                    "kernel": "fa_fwd_sm103_kernel<%d,%s,%s,%d,%d>" % (w.D, str(w.causal).lower(),
                                                                      str(w.varlen).lower(),
                                                                      1 if w.window is not None else 0, w.Dv)}

    # Two more denominators for the tensor-bound kernels: the nominal dense BF16
    # peak of one GB300 (2.25 PFLOP/s: NVIDIA's 36 PFLOP/s for eight GPUs is
    # quoted with 2:4 sparsity) and the clock-derived ceiling, SMs x 8192
    # dense BF16 FLOP per clock and SM x the median SM clock of the timed run.
    clk = clocks.summary()
    if roofline.get("bound") == "tensor":
        nominal = NOMINAL_BF16_TFLOPS * (2.0 if w.fp8 else 1.0)
        roofline["nominal_peak"] = nominal
        roofline["frac_of_nominal"] = roofline["achieved"] / nominal
        if clk.get("sm_mhz"):
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            ceiling = sms * 8192 * (2 if w.fp8 else 1) * clk["sm_mhz"] * 1e6 / 1e12
            roofline["clock_ceiling"] = ceiling
            roofline["frac_of_clock_ceiling"] = roofline["achieved"] / ceiling

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, desc, _ = cpu_oracle_rate(w, host_inputs, args.cpu_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "e4m3" if w.fp8 else "bf16", "data": "synthetic",
                "step_ms": step_stats,
                "config": workload_config(w, world), "l2": l2_note, "sustained": sustained,
                "frac_of_peak": value / world / peak,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
