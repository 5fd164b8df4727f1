"""Benchmark of fused RMSNorm+MatMul on GB300 through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--shapes all|none] [--no-cpu-baseline]

One step = one rmsnorm_matmul() call over one batch of the workload (the whole
hot path: gain, row statistic, contraction, scaled epilogue, all in one
kernel).  Default workload: decode-time QKV projection, X [16,4096], W
[4096,6144] (HBM-bound on W).  The headline value is HBM GB/s of algorithmic
traffic (X + W + Y bytes, each moved once) over the device time of exactly K
steps.

Timing: the K steps are captured as back-to-back calls in CUDA graphs on one
stream and replayed once, bracketed by CUDA events on that stream, after W
untimed warm-up calls.  Cold L2: every step reads its own copy of X, g, W and
writes its own Y; the copies rotate and together exceed 3x the L2 size, so no
step finds its inputs in L2.  SM clocks and throttle reasons are sampled with
nvidia-smi during the timed region.

Also reported on the same JSON line: a roofline object for the fused kernel,
an end-to-end number through the C ABI from pinned host buffers (host->device
copies of X, g and W and the device->host copy of Y inside the timed region),
the fp64 CPU oracle timed on the host cores (cpu_baseline), and per-shape
results for all five workloads.

--impl reference times the fp64 CPU oracle (the only reference available:
the pages ship no code) on the same workload and prints the same JSON line
with "impl": "reference".

Multi-GPU: the operation has no exchange step at this size, so N GPUs run N
independent replicas (weak scaling); a gloo barrier brackets the timed region
and rank 0 reports the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RMSNorm+MatMul TFLOP/s & HBM GB/s, % of GB300 roofline, per shape"
DEFAULT_WORKLOAD = "decode_qkv_16x4096x6144"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"

    def find(obj, key):
        if isinstance(obj, dict):
            if key in obj and isinstance(obj[key], (int, float)):
                return float(obj[key])
            for v in obj.values():
                r = find(v, key)
                if r is not None:
                    return r
        return None

    out = {}
    for k in FALLBACK_PEAKS:
        v = find(d, k)
        out[k] = v if v is not None else FALLBACK_PEAKS[k]
    return out, "measured"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


class RankSync:
    """Barrier and max-over-ranks for N replicas (one process per GPU).

    The operation has no exchange step, so N GPUs run N independent replicas;
    the only communication is this host-side barrier and the MAX of the
    per-rank timings, over a gloo process group (no NCCL, no data-path
    collective).  With one rank every call is a no-op.
    """

    def __init__(self, dist):
        self.dist = dist

    @classmethod
    def create(cls, world_size: int):
        if world_size <= 1:
            return cls(None)
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return cls(dist)

    def __call__(self, val=None):
        """Barrier; with a value, return the maximum of it over all ranks."""
        if self.dist is None:
            return val
        if val is None:
            self.dist.barrier()
            return None
        import torch
        t = torch.tensor([float(val)], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.barrier()
            self.dist.destroy_process_group()


def whole_job_value(units_per_rank: float, world_size: int, max_secs: float) -> float:
    """Units all ranks processed per second of the slowest rank (weak scaling)."""
    return world_size * units_per_rank / max_secs


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.windows = []

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[4:]))
                    except ValueError:
                        continue
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        inside = [r for r in rows if any(a - 0.15 <= r[0] <= b + 0.15 for a, b in self.windows)]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[4][1:5])
                          if v.lower().startswith("active")})
        powers = []
        for r in use:
            try:
                powers.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons,
                "power_w": statistics.median(powers) if powers else None,
                "samples": len(use), "in_window": bool(inside)}


def traffic_from_profile(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        with open(os.path.join(ROOT, "sm_rmsnorm_matmul_gb300", "csrc", "kernels.cu"), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernels_cu_sha256_16") != h:
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------- GPU timing
def make_copies(w, n_copies, device, torch, inputs, out_cols=None, weight_nk=False):
    X, g, W = inputs.generate_workload(w)
    if weight_nk:
        W = W.t().contiguous()   # [N, K], a linear layer's layout
    Xd, gd, Wd = X.to(device), g.to(device), W.to(device)
    copies = []
    for i in range(n_copies):
        if i == 0:
            xs, gs, ws = Xd, gd, Wd
        else:
            xs, gs, ws = Xd.clone(), gd.clone(), Wd.clone()
        ys = torch.empty((w.M, out_cols or w.N), dtype=torch.bfloat16, device=device)
        copies.append((xs, gs, ws, ys))
    return (X, g, W), copies


def n_rotating_copies(w, l2_bytes):
    per = w.bytes_algorithmic
    return max(1, math.ceil(3 * l2_bytes / per) + 1) if per < 3 * l2_bytes else 1


def time_graph(torch, stream, step_fn, n_copies, K, chunk=500):
    """Capture K back-to-back steps (step i uses copy i % n_copies) in CUDA
    graphs of at most `chunk` steps, replay them once, return seconds, the
    wall-clock window and the graphs (which replay_times can run again)."""
    graphs = []
    done = 0
    while done < K:
        c = min(chunk, K - done)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(done, done + c):
                step_fn(i % n_copies)
        graphs.append(gr)
        done += c
    for gr in graphs:          # upload / first replay, untimed
        gr.replay()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for gr in graphs:
            gr.replay()
        end.record(stream)
    end.synchronize()
    t1 = time.time()
    return start.elapsed_time(end) / 1e3, (t0, t1), graphs


def replay_times(torch, stream, graphs, n):
    """Replay the captured K steps n more times; seconds of each replay."""
    out = []
    for _ in range(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for gr in graphs:
                gr.replay()
            end.record(stream)
        end.synchronize()
        out.append(start.elapsed_time(end) / 1e3)
    return out


def bench_workload(torch, rmm, inputs, w, K, W_warm, device, stream, l2, with_unfused=True,
                   sampler=None, barrier=None, gated=False, weight_nk=False, lora_r=0, replays=0,
                   folded=False):
    """gated: time the gated form (Y [M, N/2]); weight_nk: W stored [N, K];
    lora_r > 0: the low-rank adapter form with rank lora_r; folded: the gain
    folded into W once before timing (fold_gain), then rmsnorm_matmul_folded
    per step; replays > 0: replay
    the timed steps that many more times (reported beside the timed run, which
    alone gives the result)."""
    n_copies = n_rotating_copies(w, l2)
    F = w.N // 2
    host, copies = make_copies(w, n_copies, device, torch, inputs, out_cols=F if gated else None,
                               weight_nk=weight_nk)
    if lora_r:
        A, B = (t.to(device) for t in inputs.lora_adapter(w.K, w.N, lora_r, seed=w.seed + 100))
    wgs = [rmm.fold_gain(c[1], c[2]) for c in copies] if folded else None

    def step(i):
        x, g, wt, y = copies[i]
        if folded:
            rmm.rmsnorm_matmul_folded(x, wgs[i], w.eps, out=y, stream=stream)
        elif lora_r:
            rmm.rmsnorm_matmul_lora(x, g, wt, A, B, w.eps, out=y, stream=stream)
        elif gated or weight_nk:
            rmm.rmsnorm_matmul_ex(x, g, wt, w.eps, weight_nk=weight_nk, gated=gated, out=y, stream=stream)
        else:
            rmm.rmsnorm_matmul(x, g, wt, w.eps, out=y, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(W_warm, 1)):
            step(i % n_copies)
    stream.synchronize()
    if rmm.device_status(stream) != 0:
        raise RuntimeError("device status not clean after warm-up")
    if barrier:
        barrier()
    torch.cuda.synchronize()
    secs, window, graphs = time_graph(torch, stream, step, n_copies, K)
    torch.cuda.synchronize()
    if barrier:
        secs = barrier(secs)
    if sampler:
        sampler.mark(*window)
    extra = replay_times(torch, stream, graphs, replays) if replays else []
    status = rmm.device_status(stream)
    del graphs
    res = {"secs": secs, "n_copies": n_copies, "status": status, "host": host, "replays": [secs] + extra,
           "copies": copies, "path": 1 if gated else rmm.dispatch_path(w.M, w.K, w.N),
           "plan": rmm.describe_plan(w.M, w.K, w.N, gated=gated)}
    if with_unfused:
        xn = [torch.empty((w.M, w.K), dtype=torch.bfloat16, device=device) for _ in range(n_copies)]
        zs = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device) for _ in range(n_copies)] \
            if gated or lora_r else None
        ts = torch.empty((w.M, lora_r), dtype=torch.bfloat16, device=device) if lora_r else None

        def step_unfused(i):
            # the separate kernels: RMSNorm, MatMul (and, gated, torch's
            # elementwise silu(gate) * up on the bf16 product; with an
            # adapter, Xn @ A, T @ B and torch's elementwise add)
            x, g, wt, y = copies[i]
            rmm.rmsnorm(x, g, w.eps, out=xn[i], stream=stream)
            if lora_r:
                rmm.matmul(xn[i], wt, out=y, stream=stream)
                rmm.matmul(xn[i], A, out=ts, stream=stream)
                rmm.matmul(ts, B, out=zs[i], stream=stream)
                with torch.cuda.stream(stream):
                    y.add_(zs[i])
            elif gated:
                rmm.matmul(xn[i], wt, out=zs[i], stream=stream)
                with torch.cuda.stream(stream):
                    torch.mul(torch.nn.functional.silu(zs[i][:, :F]), zs[i][:, F:], out=y)
            else:
                rmm.matmul(xn[i], wt, out=y, stream=stream)

        with torch.cuda.stream(stream):
            for i in range(2):
                step_unfused(i % n_copies)
        stream.synchronize()
        ku = max(1, min(K, 200))
        s_unf, _, g2 = time_graph(torch, stream, step_unfused, n_copies, ku)
        res["unfused_secs_per_step"] = s_unf / ku
        del g2, xn, zs, ts
    return res


def bench_attention(torch, rmm, inputs, w, K, device, stream, l2, sampler=None):
    """Time qknorm_attention on one AttentionWorkload: K back-to-back calls in
    CUDA graphs, each on its own copy of the fused QKV tensor (copies rotate
    so that every call misses L2), and torch's rms_norm + scaled dot-product
    attention on the same inputs as context."""
    per = w.bytes_algorithmic
    n_copies = max(1, math.ceil(3 * l2 / per) + 1) if per < 3 * l2 else 1
    qkv, gq, gk = inputs.attention_inputs(w.B, w.S, w.Hq, w.Hkv, w.D, w.seed)
    gq, gk = gq.to(device), gk.to(device)
    copies = []
    for _ in range(n_copies):
        t = qkv.to(device)
        o = torch.empty((w.B, w.S, w.Hq, w.D), dtype=torch.bfloat16, device=device)
        copies.append((inputs.split_qkv(t, w.B, w.S, w.Hq, w.Hkv, w.D), o))

    def step(i):
        (q, k, v), o = copies[i]
        rmm.qknorm_attention(q, k, v, gq, gk, w.eps, causal=w.causal, out=o, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i % n_copies)
    stream.synchronize()
    if rmm.device_status(stream) != 0:
        raise RuntimeError("device status not clean after warm-up")
    secs, window, graphs = time_graph(torch, stream, step, n_copies, K)
    if sampler:
        sampler.mark(*window)
    del graphs
    status = rmm.device_status(stream)
    F = torch.nn.functional

    def step_torch(i):
        (q, k, v), _ = copies[i]
        qn = F.rms_norm(q, (w.D,), gq, w.eps)
        kn = F.rms_norm(k, (w.D,), gk, w.eps)
        F.scaled_dot_product_attention(qn.transpose(1, 2), kn.transpose(1, 2), v.transpose(1, 2),
                                       is_causal=w.causal, enable_gqa=True)

    unfused = None
    try:
        with torch.cuda.stream(stream):
            for i in range(2):
                step_torch(i % n_copies)
        ku = max(3, K // 4)
        s_u, _, g2 = time_graph(torch, stream, step_torch, n_copies, ku)
        del g2
        unfused = s_u / ku
    except (RuntimeError, TypeError):   # an older torch without enable_gqa or rms_norm
        unfused = None
    del copies
    return {"secs": secs, "n_copies": n_copies, "status": status, "unfused_secs_per_step": unfused,
            "l2": (f"rotating input/output copies: {n_copies} x {per / 1e6:.1f} MB > 3 x L2 "
                   f"({l2 / 1e6:.0f} MB)") if n_copies > 1 else
                  f"inputs ({per / 1e6:.0f} MB) larger than L2 ({l2 / 1e6:.0f} MB)"}


def attention_entry(w, t, r, peaks, k):
    tflops = w.flops / t / 1e12
    e = {"workload": w.name + " (QK-normalised attention)", "path": "qknorm_attention (tcgen05)",
         "steps": k, "us_per_call": round(t * 1e6, 3), "tflops": round(tflops, 2),
         "hbm_gbs": round(w.bytes_algorithmic / t / 1e9, 1), "bound": "tensor",
         "roofline_frac": round(tflops / peaks["bf16_tflops"], 4),
         "frac_of_tensor_peak_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4),
         "copies": r["n_copies"], "l2": r["l2"], "device_status": r["status"]}
    if r.get("unfused_secs_per_step"):
        e["torch_rms_norm_sdpa_us"] = round(r["unfused_secs_per_step"] * 1e6, 3)
    return e


def e2e_bench(torch, rmm, w, host, device, stream, K):
    """Pinned host X, g, W -> device, fused call, Y -> pinned host, per step."""
    X, g, W = host
    hX, hg, hW = X.pin_memory(), g.pin_memory(), W.pin_memory()
    hY = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    dX = torch.empty_like(hX, device=device)
    dg = torch.empty_like(hg, device=device)
    dW = torch.empty_like(hW, device=device)
    dY = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)

    def step():
        with torch.cuda.stream(stream):
            dX.copy_(hX, non_blocking=True)
            dg.copy_(hg, non_blocking=True)
            dW.copy_(hW, non_blocking=True)
            rmm.rmsnorm_matmul(dX, dg, dW, w.eps, out=dY, stream=stream)
            hY.copy_(dY, non_blocking=True)

    for _ in range(3):
        step()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
    for _ in range(K):
        step()
    with torch.cuda.stream(stream):
        end.record(stream)
    end.synchronize()
    secs = start.elapsed_time(end) / 1e3
    h2d = (hX.numel() + hg.numel() + hW.numel()) * 2
    d2h = hY.numel() * 2
    return secs, h2d, d2h


# ----------------------------------------------------------- CPU reference
def cpu_oracle_run(w, budget_s, steps=None, warmup=0):
    """Time the fp64 oracle on host cores.  Returns (secs_per_step, bytes per
    step, sample description, threads).  With `steps`, runs exactly that many
    steps, each on a row sample sized so the whole run fits the budget."""
    import numpy as np
    import oracle
    from sm_rmsnorm_matmul_gb300 import inputs
    X, g, W = inputs.generate_workload(w)
    Xf, gf, Wf = oracle.to_f64(X), oracle.to_f64(g), oracle.to_f64(W)
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    # probe: one row block to estimate the cost per row
    probe_rows = min(w.M, max(1, threads))
    t = time.perf_counter()
    oracle.rmsnorm_matmul(Xf[:probe_rows], gf, Wf, w.eps, lib=lib)
    per_row = (time.perf_counter() - t) / probe_rows
    total_steps = steps if steps is not None else None
    if total_steps is None:
        rows = w.M if per_row * w.M <= budget_s else max(1, int(budget_s / per_row))
        rows = min(rows, w.M)
        reps = max(1, int(budget_s / max(per_row * rows, 1e-6)))
    else:
        rows_fit = int(budget_s / max(per_row * total_steps, 1e-9))
        rows = max(1, min(w.M, rows_fit))
        reps = total_steps
    rows = max(1, min(rows, w.M))
    idx = inputs.sample_rows(w.M, rows) if rows < w.M else list(range(w.M))
    Xs = np.ascontiguousarray(Xf[idx])
    for _ in range(warmup):
        oracle.rmsnorm_matmul(Xs, gf, Wf, w.eps, lib=lib)
    t = time.perf_counter()
    for _ in range(reps):
        oracle.rmsnorm_matmul(Xs, gf, Wf, w.eps, lib=lib)
    secs = (time.perf_counter() - t) / reps
    nbytes = 2 * (len(idx) * w.K + w.K * w.N + len(idx) * w.N)
    sample = (f"{len(idx)} of {w.M} rows x all {w.N} columns, {reps} repetitions, "
              f"fp64 oracle, {threads} OpenMP threads")
    return secs, nbytes, sample, threads, len(idx), reps


def cpu_oracle_table(one_thread_secs: float = 2.0):
    """The fp64 oracle on every workload, on the host cores: all rows of the
    workloads up to 4096 rows, the 256-row sample of the larger one (its
    full-size time extrapolated from the sample, and labelled so), with every
    OpenMP thread, and with one thread on a row sample of about
    `one_thread_secs`."""
    import numpy as np
    import oracle
    from sm_rmsnorm_matmul_gb300 import inputs
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    rows_out = []
    for name in inputs.WORKLOAD_ORDER:
        w = inputs.WORKLOADS[name]
        X, g, W = inputs.generate_workload(w)
        Xf, gf, Wf = oracle.to_f64(X), oracle.to_f64(g), oracle.to_f64(W)
        del X, W
        full = w.M <= 4096
        idx = list(range(w.M)) if full else inputs.sample_rows(w.M, 256)
        Xs = np.ascontiguousarray(Xf[idx])
        t = time.perf_counter()
        oracle.rmsnorm_matmul(Xs, gf, Wf, w.eps, lib=lib)
        secs = time.perf_counter() - t
        flops = 2.0 * len(idx) * w.K * w.N
        per_row_one = secs * threads / len(idx)       # estimate for one thread
        n1 = max(1, min(len(idx), int(one_thread_secs / max(per_row_one, 1e-9))))
        idx1 = inputs.sample_rows(w.M, n1) if n1 < w.M else list(range(w.M))
        X1 = np.ascontiguousarray(Xf[idx1])
        t = time.perf_counter()
        oracle.rmsnorm_matmul(X1, gf, Wf, w.eps, nthreads=1, lib=lib)
        s1 = time.perf_counter() - t
        e = {"workload": name, "rows": len(idx), "rows_of": w.M, "threads": threads,
             "secs": round(secs, 4), "gflops_f64": round(flops / secs / 1e9, 2),
             "one_thread": {"rows": len(idx1), "secs": round(s1, 4),
                            "gflops_f64": round(2.0 * len(idx1) * w.K * w.N / s1 / 1e9, 2)}}
        if not full:
            e["full_size_secs_extrapolated"] = round(secs * w.M / len(idx), 2)
        rows_out.append(e)
        del Xf, Wf, Xs, X1
    return {"nproc": os.cpu_count(), "openmp_threads": threads, "kind": "oracle",
            "workloads": rows_out}


# ---------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--shapes", choices=["all", "none"], default="all")
    ap.add_argument("--form", choices=["fused", "folded"], default="fused",
                    help="the timed call: rmsnorm_matmul, or rmsnorm_matmul_folded on a W with the "
                         "gain folded in once before timing (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--reference-budget", type=float, default=90.0,
                    help="seconds of oracle work for the whole --impl reference run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from sm_rmsnorm_matmul_gb300 import inputs
    ws, rank, local = dist_env()
    if args.workload in inputs.ATTENTION_WORKLOADS:
        # one attention line alone (profiling and quick checks)
        return run_attention_only(args, inputs.ATTENTION_WORKLOADS[args.workload], rank)
    w = inputs.WORKLOADS[args.workload] if args.workload in inputs.WORKLOADS else inputs.PROFILE_CASES[args.workload]

    if args.impl == "reference":
        return run_reference(args, w, ws, rank)

    import torch
    import sm_rmsnorm_matmul_gb300 as rmm
    rmm.lib()  # fail loudly if the CUDA library is missing

    sync = RankSync.create(ws)
    barrier = sync if ws > 1 else None

    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    gpu_id = None
    try:
        gpu_id = f"GPU-{props.uuid}"
    except Exception:  # noqa: BLE001
        pass
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)

    with ClockSampler(gpu_id) as sampler:
        main_res = bench_workload(torch, rmm, inputs, w, args.steps, args.warmup, device,
                                  stream, l2, with_unfused=True, sampler=sampler,
                                  barrier=barrier, replays=4 if ws == 1 else 0,
                                  folded=args.form == "folded")
        host = main_res["host"]
        e2e_steps = max(3, min(args.steps, 200))
        e2e_secs, h2d, d2h = e2e_bench(torch, rmm, w, host, device, stream, e2e_steps)
        if ws > 1:
            e2e_secs = sync(e2e_secs)
        del main_res["copies"]
        shapes = []
        if args.shapes == "all" and rank == 0:
            for name in inputs.WORKLOAD_ORDER:
                ww = inputs.WORKLOADS[name]
                est = max(ww.flops / (peaks["bf16_tflops"] * 1e12),
                          ww.bytes_xwy / (peaks["hbm_gbs"] * 1e9))
                k = int(min(5000, max(20, 0.2 / max(est, 1e-7))))
                r = bench_workload(torch, rmm, inputs, ww, k, 3, device, stream, l2,
                                   with_unfused=True, sampler=sampler)
                t = r["secs"] / k
                shapes.append(shape_entry(ww, t, r, peaks, k))
                del r
                torch.cuda.empty_cache()
            # the gated MLP on top (rmsnorm_matmul_swiglu), on the gate|up shape
            # and on a prefill-sized one
            gated_prefill = inputs.Workload(name="prefill_gatedmlp_4096x4096x28672", M=4096, K=4096,
                                            N=28672, eps=1e-5, seed=6, w_std=1 / 64, x_kind="row_scaled")
            for ww in (inputs.WORKLOADS["decode_gatedmlp_64x4096x28672"], gated_prefill):
                est = max(ww.flops / (peaks["bf16_tflops"] * 1e12),
                          gated_bytes(ww) / (peaks["hbm_gbs"] * 1e9))
                k = int(min(5000, max(20, 0.2 / max(est, 1e-7))))
                r = bench_workload(torch, rmm, inputs, ww, k, 3, device, stream, l2,
                                   with_unfused=True, sampler=sampler, gated=True)
                shapes.append(shape_entry(ww, r["secs"] / k, r, peaks, k, gated=True))
                del r
                torch.cuda.empty_cache()
            # weights stored [N, K] (a linear layer's layout, read K-major)
            for name in ("decode_qkv_16x4096x6144", "prefill_qkv_4096x4096x6144"):
                ww = inputs.WORKLOADS[name]
                est = max(ww.flops / (peaks["bf16_tflops"] * 1e12), ww.bytes_xwy / (peaks["hbm_gbs"] * 1e9))
                k = int(min(5000, max(20, 0.2 / max(est, 1e-7))))
                r = bench_workload(torch, rmm, inputs, ww, k, 3, device, stream, l2,
                                   with_unfused=False, sampler=sampler, weight_nk=True)
                e = shape_entry(ww, r["secs"] / k, r, peaks, k)
                e["workload"] += " (W stored [N, K])"
                shapes.append(e)
                del r
                torch.cuda.empty_cache()
            # the gain folded into the weights once (inference weights), then
            # one kernel per call that reads raw X
            for name in ("decode_qkv_16x4096x6144", "prefill_qkv_4096x4096x6144",
                         "large_prefill_16384x8192x8192"):
                ww = inputs.WORKLOADS[name]
                est = max(ww.flops / (peaks["bf16_tflops"] * 1e12), ww.bytes_xwy / (peaks["hbm_gbs"] * 1e9))
                k = int(min(5000, max(20, 0.2 / max(est, 1e-7))))
                r = bench_workload(torch, rmm, inputs, ww, k, 3, device, stream, l2,
                                   with_unfused=True, sampler=sampler, folded=True)
                e = shape_entry(ww, r["secs"] / k, r, peaks, k)
                e["workload"] += " (gain folded into W once)"
                e["path"] = "256-row kernel, row statistic in-kernel" if ww.M > 128 else e["path"] + ", gain of ones"
                shapes.append(e)
                del r
                torch.cuda.empty_cache()
            # the low-rank adapter form
            for name, lora_rank in (("decode_qkv_16x4096x6144", 16), ("prefill_qkv_4096x4096x6144", 64)):
                ww = inputs.WORKLOADS[name]
                est = max(ww.flops / (peaks["bf16_tflops"] * 1e12), ww.bytes_xwy / (peaks["hbm_gbs"] * 1e9))
                k = int(min(5000, max(20, 0.2 / max(est, 1e-7))))
                r = bench_workload(torch, rmm, inputs, ww, k, 3, device, stream, l2,
                                   with_unfused=True, sampler=sampler, lora_r=lora_rank)
                shapes.append(shape_entry(ww, r["secs"] / k, r, peaks, k, lora_r=lora_rank))
                del r
                torch.cuda.empty_cache()
            # QK-normalised attention over the prefill QKV projection's output
            for aw in inputs.ATTENTION_WORKLOADS.values():
                k = int(min(2000, max(20, 0.3 / (aw.flops / (peaks["bf16_tflops"] * 1e12) * 3))))
                r = bench_attention(torch, rmm, inputs, aw, k, device, stream, l2, sampler=sampler)
                shapes.append(attention_entry(aw, r["secs"] / k, r, peaks, k))
                del r
                torch.cuda.empty_cache()
    clocks = sampler.summary()

    K = args.steps
    t_step = main_res["secs"] / K
    bytes_step = w.bytes_xwy
    value = whole_job_value(bytes_step, ws, t_step) / 1e9
    achieved = w.bytes_algorithmic / t_step / 1e9
    bound = "hbm" if w.flops / w.bytes_xwy < 290 else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        tf = w.flops / t_step / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4)}
    roof["traffic"] = traffic_from_profile(w.name)
    roof["peak_source"] = peak_src
    roof["kernel"] = (kernel_name(rmm, w) if args.form == "fused" or w.M <= 128
                      else "tall_kernel<row statistic> (gain folded into W)")
    roof["algorithmic_bytes_per_launch"] = w.bytes_algorithmic

    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t_step * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; see sm_rmsnorm_matmul_gb300/inputs.py)",
        "config": {
            "workload": w.name, "M": w.M, "K": w.K, "N": w.N, "eps": w.eps, "seed": w.seed,
            "accumulate": "fp32", "path": "small-M (gemv)" if main_res["path"] == 2 else "row-tile",
            "plan": main_res["plan"],
            "l2": f"rotating input/output copies: {main_res['n_copies']} x "
                  f"{w.bytes_algorithmic / 1e6:.1f} MB > 3 x L2 ({l2 / 1e6:.0f} MB)"
                  if main_res["n_copies"] > 1 else
                  f"inputs ({w.bytes_algorithmic / 1e6:.0f} MB) larger than L2 ({l2 / 1e6:.0f} MB)",
            "timing": "CUDA graphs of back-to-back C-ABI calls, CUDA events on the launch stream",
            "form": "rmsnorm_matmul" if args.form == "fused" else
                    "rmsnorm_matmul_folded (gain folded into W once, before timing)",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "tflops": round(w.flops / t_step / 1e12, 2),
        "roofline": roof,
        "roofline_time_frac": round(max(w.flops / (peaks["bf16_tflops"] * 1e12),
                                        w.bytes_xwy / (peaks["hbm_gbs"] * 1e9)) / t_step, 4),
        "unfused_pair_ms_per_step": round(main_res["unfused_secs_per_step"] * 1e3, 6),
        "e2e": {"value": round(ws * bytes_step / (e2e_secs / e2e_steps) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_secs / e2e_steps * 1e3, 4), "steps": e2e_steps},
        "gpu_launches": K,
        # the same K steps replayed again (the timed run first): spread of the measurement
        "graph_replays": {"count": len(main_res["replays"]),
                          "median_ms_per_step": round(statistics.median(main_res["replays"]) / K * 1e3, 6),
                          "min_ms_per_step": round(min(main_res["replays"]) / K * 1e3, 6),
                          "max_ms_per_step": round(max(main_res["replays"]) / K * 1e3, 6)},
        "clocks": clocks,
        "device_status": main_res["status"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        secs, nbytes, sample, threads, _, _ = cpu_oracle_run(w, args.cpu_budget)
        out["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s",
                               "cores": threads, "kind": "oracle", "sample": sample,
                               "secs_per_call": round(secs, 4)}
        if args.shapes == "all":
            out["cpu_oracle_table"] = cpu_oracle_table()
    if shapes:
        out["shapes"] = shapes
        # compact copies of every line, last on the line (a reader that keeps
        # only its tail still sees each workload's result)
        out["other_lines"] = [compact(e) for e in shapes if e["workload"] not in inputs.WORKLOADS]
        out["per_config"] = [compact(e) for e in shapes if e["workload"] in inputs.WORKLOADS]
    if rank == 0:
        print(json.dumps(out), flush=True)
    sync.close()


def run_attention_only(args, aw, rank):
    """`--workload <attention workload>`: time qknorm_attention alone for
    --steps calls and print its shape entry as one JSON line."""
    import torch
    import sm_rmsnorm_matmul_gb300 as rmm
    from sm_rmsnorm_matmul_gb300 import inputs
    rmm.lib()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    peaks, _ = load_peaks()
    stream = torch.cuda.Stream(device=device)
    r = bench_attention(torch, rmm, inputs, aw, args.steps, device, stream, l2)
    e = attention_entry(aw, r["secs"] / args.steps, r, peaks, args.steps)
    if rank == 0:
        print(json.dumps(e), flush=True)


def kernel_name(rmm, w):
    """Name of the kernel the fused call launches for this workload."""
    plan = rmm.describe_plan(w.M, w.K, w.N)
    if plan["path"] == 2:
        return f"gemv_kernel<fused> ({plan['splits']} K pieces per 64-column unit)"
    if plan["cluster"]:
        bn = -(-w.N // plan["tiles"]) if plan["tiles"] else 256
        width = ", 128-column tiles" if bn <= 128 else ""
        return f"rows_kernel<fused, K split x{plan['splits']} in a cluster{width}>"
    if w.M > 128:
        return "rows_ta_kernel (A operand in tensor memory)"
    return "rows_kernel<fused>"


def compact(e):
    """A short form of one shape entry: time, rates, fraction of its roofline
    (of the measured burst peak) and, where timed, the unfused kernels' time."""
    c = {"w": e["workload"].replace(" (", "(")[:48], "us": round(e["us_per_call"], 2), "tf": round(e["tflops"], 1),
         "gbs": round(e["hbm_gbs"]), "frac": round(e["roofline_frac"], 3), "of": e["bound"]}
    for k in ("unfused_pair_us", "unfused_us", "torch_rms_norm_sdpa_us"):
        if k in e:
            c["unf_us"] = round(e[k], 1)
    return c


def gated_bytes(w):
    """X + W + Y bytes of the gated form (Y has N/2 columns)."""
    return 2 * (w.M * w.K + w.K * w.N + w.M * (w.N // 2))


def shape_entry(w, t, r, peaks, k, gated=False, lora_r=0):
    nbytes = gated_bytes(w) if gated else w.bytes_xwy
    flops = w.flops
    if lora_r:   # + A and B; + (X*g) @ A and T @ B (the intermediate T is not algorithmic)
        nbytes += 2 * (w.K * lora_r + lora_r * w.N)
        flops += 2 * w.M * lora_r * (w.K + w.N)
    tflops = flops / t / 1e12
    gbs = nbytes / t / 1e9
    roof_t = max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    bound = "tensor" if flops / (peaks["bf16_tflops"] * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"
    e = {"workload": w.name + (" (gated: silu(gate) * up)" if gated else "") +
         (f" (low-rank adapter, R = {lora_r})" if lora_r else ""),
         "path": "small-M (gemv)" if r["path"] == 2 else "row-tile",
         "plan": r.get("plan"),
         "steps": k, "us_per_call": round(t * 1e6, 3), "tflops": round(tflops, 2),
         "hbm_gbs": round(gbs, 1), "bound": bound, "roofline_frac": round(roof_t / t, 4),
         "copies": r["n_copies"], "device_status": r["status"]}
    if bound == "tensor":
        e["frac_of_tensor_peak_sustained"] = round(tflops / peaks["bf16_tflops_sustained"], 4)
    if "unfused_secs_per_step" in r:
        e["unfused_us" if gated or lora_r else "unfused_pair_us"] = round(r["unfused_secs_per_step"] * 1e6, 3)
    return e


def run_reference(args, w, ws, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    budget = args.reference_budget
    K, Wm = args.steps, args.warmup
    # W untimed warm-up steps, then exactly K timed steps, each on a row sample
    # sized so that the whole run stays within the budget
    secs, nbytes, sample, threads, rows, reps = cpu_oracle_run(w, budget / (1 + Wm / max(K, 1)),
                                                               steps=K, warmup=Wm)
    value = nbytes / secs / 1e9
    out = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": K, "warmup": Wm, "ms_per_step": round(secs * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; see sm_rmsnorm_matmul_gb300/inputs.py)",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "eps": w.eps,
                   "seed": w.seed, "reference": "fp64 CPU oracle (oracle/rmm_oracle.c); "
                   "the pages ship no implementation"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main() or 0)
