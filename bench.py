#!/usr/bin/env python3
"""Benchmark of the GB300 exact-attention forward.

One step = one ``attn_fwd`` call (the whole hot path: TMA loads, QK^T and P.V on the tensor cores,
online softmax, O/LSE stores) over the long-context workload B=1, Hq=32, Hkv=8, N=32768, D=128,
causal, bf16 (FLOPs = 4*B*Hq*N^2*D / 2).  Inputs (402 MB) and the output (268 MB) exceed the
129 MB L2, so steps run back to back without an explicit flush.  The context legs (the five
configurations at N = 128..4096, the other long lengths, wide heads, split-KV, the backward and
the MLA decode) follow in the same line; those whose inputs fit in L2 are timed after a 256 MB
flush before each launch.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead (bounded sample per
step, on the host cores).  Under torchrun (``--gpus N``) each rank runs an independent replica on
its own GPU; the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS and ms (causal-adjusted) at N=1K–32K; % of bf16 TC peak"
UNIT = "TFLOPS"
DEFAULT_WORKLOAD = "long-gqa8-causal-n32768"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
KERNEL_SOURCES = ["exact_attention_forward_attn_gb300/csrc/attn_fwd_kernel.cuh",
                  "exact_attention_forward_attn_gb300/csrc/attn_fwd_pair_kernel.cuh",
                  "exact_attention_forward_attn_gb300/csrc/ptx.cuh",
                  "exact_attention_forward_attn_gb300/csrc/attn_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def kernel_hash() -> str:
    """Hash of the forward's sources with comments and whitespace removed, so that the stored
    DRAM traffic stays attached to the code it was measured on, not to its comments."""
    import re

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                 # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel build."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_sha") != kernel_hash():
        return None
    key = f"bytes_per_launch[{workload_name}]"
    return float(kv[key]) if key in kv else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def physical_gpu_index(local: int):
    """nvidia-smi index of CUDA device `local` (honours a numeric CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over the ranks of the default process group (the value itself when
    there is none).  NCCL needs a CUDA tensor; gloo (the CPU tests) a CPU one."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job rate of independent replicas: every rank's units over the slowest rank's time
    (weak scaling: each rank processes the same amount of work)."""
    return units_per_rank * world / max_seconds


def cpu_sample_rows(w, n_rows_per_head):
    """Seeded query rows for the CPU oracle's bounded sample (same rows for every head)."""
    import torch

    n_rows_per_head = min(n_rows_per_head, w.N)
    g = torch.Generator().manual_seed(9000 + w.N)
    rows = torch.randperm(w.N, generator=g)[:n_rows_per_head].sort().values.to(torch.int32)
    return rows.view(1, 1, -1).expand(w.B, w.Hq, -1).contiguous()


def sample_flops(w, rows) -> float:
    """FLOPs of the oracle's work on the sampled rows (4*D per visible key)."""
    vis = (rows.long() + 1).sum().item() if w.causal else rows.numel() * w.N
    return 4.0 * w.D * float(vis)


def time_oracle(w, q, k, v, seconds_target: float, max_rows: int = 4096):
    """Calibrate the number of sampled rows per head so one oracle call takes ~seconds_target."""
    import oracle

    rows = cpu_sample_rows(w, 8)
    t0 = time.perf_counter()
    oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    dt = max(time.perf_counter() - t0, 1e-3)
    rate = sample_flops(w, rows) / dt
    n = int(min(max_rows, w.N, max(8, 8 * seconds_target / dt)))
    return n, rate


def causal_work(w, rows=None) -> float:
    """Visible (query, key) pairs of workload w, over all rows or over the sampled `rows`
    [B, Hq, R] (under the causal mask row i sees i + 1 keys)."""
    if rows is None:
        per_head = w.N * (w.N + 1) / 2 if w.causal else float(w.N) * w.N
        return per_head * w.B * w.Hq
    if w.causal:
        return float((rows.long() + 1).sum().item())
    return float(rows.numel()) * w.N


def _parity(o_gpu, l_gpu, o_ref, l_ref):
    """max|dO|, max|dLSE| and whether every element is within the tolerance of the tests
    (|dO| <= 2e-2 + 2e-2 |O_ref|, |dLSE| <= 1e-3)."""
    import numpy as np

    o = o_gpu.float().numpy().astype(np.float64)
    l = l_gpu.numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    lerr = np.abs(l - l_ref)
    ok = bool(np.all(np.isfinite(o)) and not (err > 2e-2 + 2e-2 * np.abs(o_ref)).any()
              and lerr.max() <= 1e-3)
    return {"max_abs_dO": float(err.max()), "max_abs_dLSE": float(lerr.max()),
            "within_tolerance": ok}


def cpu_baseline_table(gpu_us=None, gpu_out=None):
    """The oracle as it stands, timed on the host cores at all cores and at one core: the five
    configurations in full (one-core C3, 0.27 TFLOP, on 128 seeded rows per head, extrapolated),
    the long-context lengths on the 64 seeded rows per head the parity tests compare,
    extrapolated to every row by the exact work ratio (visible query-key pairs), labelled.
    Where `gpu_out` holds the GPU's O and LSE of a workload (CPU tensors; for the long lengths
    the rows the parity tests sample), the all-core run's results are also compared with them."""
    import oracle
    from exact_attention_forward_attn_gb300 import workloads as wl

    all_cores = oracle.default_threads()
    table = []

    def timed(fn, repeats):
        ts = []
        for _ in range(repeats):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return statistics.median(ts)

    for w in (wl.TINY_NONCAUSAL, wl.TINY_CAUSAL, wl.GQA4_CAUSAL, wl.GQA8_CAUSAL, wl.MHA,
              wl.MHA_OUTLIER, wl.MQA, *wl.LONG.values()):
        q, k, v = wl.make_qkv(w)
        entry = {"workload": w.name, "gflop": w.flops / 1e9}
        for label, threads in (("all_cores", all_cores), ("one_core", 1)):
            long_cfg = w.N > 4096
            if long_cfg or (threads == 1 and w.flops > 1e11):
                rows = wl.sample_rows(w, 64 if long_cfg else 128)
                res = {}
                dt = timed(lambda: res.setdefault(0, oracle.attn_ref(
                    q, k, v, w.causal, w.sm_scale, rows=rows.numpy(), n_threads=threads)), 1)
                if long_cfg and threads == all_cores and gpu_out and w.name in gpu_out:
                    entry["parity_sampled_rows"] = _parity(*gpu_out[w.name], *res[0])
                scale = causal_work(w) / causal_work(w, rows)
                entry[label] = {"s": dt * scale, "kind": "extrapolated",
                                "sample": f"{rows.shape[2]} seeded rows per head, {dt:.2f} s"}
            else:
                reps = 3 if w.flops < 2e10 else 1
                res = {}
                dt = timed(lambda: res.__setitem__(0, oracle.attn_ref(
                    q, k, v, w.causal, w.sm_scale, n_threads=threads)), reps)
                entry[label] = {"s": dt, "kind": "full"}
                if threads == all_cores and gpu_out and w.name in gpu_out:
                    entry["parity"] = _parity(*gpu_out[w.name], *res[0])
            entry[label]["cores"] = threads
            entry[label]["tflops"] = w.flops / entry[label]["s"] / 1e12
        if gpu_us and w.name in gpu_us:
            entry["gpu_us"] = gpu_us[w.name]
            entry["speedup_vs_all_cores"] = entry["all_cores"]["s"] * 1e6 / gpu_us[w.name]
        table.append(entry)
    return table


def run_reference(args, w):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    import oracle
    from exact_attention_forward_attn_gb300 import workloads as wl

    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = wl.make_qkv(w)
    n_rows, _ = time_oracle(w, q, k, v, args.ref_step_seconds)
    rows = cpu_sample_rows(w, n_rows)
    flops = sample_flops(w, rows)
    for _ in range(args.warmup):
        oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    cores = oracle.default_threads()
    sample = (f"{n_rows} seeded query rows per head x {w.B * w.Hq} heads of {w.name} "
              f"({flops / 1e9:.2f} GFLOP per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, "host cores, no GPU"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, l2_note):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "D": w.D,
            "causal": w.causal, "sm_scale": w.sm_scale, "l2": l2_note,
            "inputs": "iid N(0,1) fp32 rounded to bf16, seeded"}


def timed_launches(fn, stream, n):
    """Run fn() n times back to back on `stream`; per-launch CUDA-event durations (ms)."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(n):
            fn()
            ev[i + 1].record(stream)
    stream.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]


def cold_launch_ms(fn, stream, flush, n, warm=3):
    """Median CUDA-event duration (ms) of fn() over n launches, each after `flush` was rewritten
    (a buffer larger than L2), so inputs smaller than L2 are read from DRAM every time.

    Everything is enqueued before the one synchronize: the flush keeps the device busy longer
    than the host takes to enqueue fn(), so each timed interval holds the device work alone and
    not the host's launch cost."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(warm + n)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
    stream.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev[warm:])


def run_profile_leg(args):
    """--profile for the backward or the MLA decode: warm-up, then timed launches, nothing else."""
    import ctypes

    import torch

    import exact_attention_forward_attn_gb300 as attn
    from exact_attention_forward_attn_gb300 import _lib
    from exact_attention_forward_attn_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    lib = _lib.load()
    sh = ctypes.c_void_p(stream.cuda_stream)
    if args.profile_kind == "mla":
        wm = {x.name: x for x in wl.MLA_CONFIGS}[args.workload]
        q, kv = wl.make_mla(wm, device=dev)
        o = torch.empty(wm.B, wm.H, attn.MLA_D_C, dtype=torch.bfloat16, device=dev)
        l = torch.empty(wm.B, wm.H, dtype=torch.float32, device=dev)
        n_sp = attn.mla_decode_num_splits(wm.B, wm.H, wm.T)
        need = attn.mla_decode_workspace_bytes(wm.B, wm.H, wm.T, n_sp)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

        def step():
            assert lib.attn_mla_decode(q.data_ptr(), kv.data_ptr(), o.data_ptr(), l.data_ptr(),
                                       wm.B, wm.H, wm.T, attn.MLA_D_C, attn.MLA_D_R,
                                       ctypes.c_float(wm.sm_scale), n_sp, ws.data_ptr(), need,
                                       sh) == 0
        name = wm.name
    else:
        wb = wl.BY_NAME[args.workload]
        q, k, v = (t.to(dev) for t in wl.make_qkv(wb))
        o, l = attn.attn_fwd(q, k, v, causal=wb.causal, sm_scale=wb.sm_scale)
        g = torch.Generator(device="cpu").manual_seed(77)
        do = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        need = int(lib.attn_bwd_workspace_bytes(wb.B, wb.Hq, wb.N))
        ws = torch.empty(need, dtype=torch.uint8, device=dev)

        def step():
            assert lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                l.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), wb.B, wb.Hq, wb.Hkv, wb.N, wb.D, int(wb.causal),
                                ctypes.c_float(wb.sm_scale), ws.data_ptr(), need, sh) == 0
        name = wb.name
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    t = timed_launches(step, stream, args.steps)
    if attn.device_status(dev) != 0:
        raise SystemExit("device status word reports an expired wait")
    print(json.dumps({"profile": name, "kind": args.profile_kind, "ms": t}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--profile", action="store_true",
                    help="timed launches only (no e2e, sweep, clocks or CPU baseline): for ncu")
    ap.add_argument("--profile-kind", choices=["forward", "backward", "mla"], default="forward",
                    help="with --profile: which path --workload names (backward: the three "
                         "backward kernels on a forward workload; mla: an MLA decode workload)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="target duration of the oracle's bounded CPU-baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=1.0,
                    help="target duration of one reference-arm step")
    args = ap.parse_args()
    if args.warmup < 0 or args.steps < 1:
        ap.error("--steps >= 1 and --warmup >= 0")

    from exact_attention_forward_attn_gb300 import workloads as wl

    if args.profile and args.profile_kind != "forward":
        return run_profile_leg(args)
    w = wl.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import ctypes

    import torch

    import exact_attention_forward_attn_gb300 as attn
    from exact_attention_forward_attn_gb300 import _lib

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    q, k, v = (t.to(dev) for t in wl.make_qkv(w))
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale, out=out, lse=lse)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if attn.device_status(dev) != 0:
        raise SystemExit("device status word reports an expired wait during warm-up")

    if args.profile:
        t = timed_launches(step, stream, args.steps)
        print(json.dumps({"profile": w.name, "ms": t}), flush=True)
        return 0

    # ---- timed region: K steps, barrier + synchronize on both sides, max over ranks ----------
    sampler = ClockSampler(physical_gpu_index(local))
    with sampler:
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        launch_ms = timed_launches(step, stream, args.steps)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
    total_ms = max_over_ranks(sum(launch_ms), dev)
    if attn.device_status(dev) != 0:
        raise SystemExit("device status word reports an expired wait in the timed region")
    clocks = sampler.summary()

    ms_per_step = total_ms / args.steps
    value = job_throughput(w.flops * args.steps, world, total_ms * 1e-3) / 1e12
    mean_launch_ms = statistics.mean(launch_ms)
    achieved = w.flops / (mean_launch_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    roofline = {
        "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
        "frac": achieved / peak, "traffic": load_traffic(w.name),
        "peak_source": f"{peak_src} bf16 dense (burst)",
        "frac_of_sustained": achieved / peak_sus,
        "hbm_gbs_algorithmic": w.bytes / (mean_launch_ms * 1e-3) / 1e9,
    }

    # ---- end to end through the public API: pinned host buffers, copies inside the region -----
    # Every step copies its inputs host->device and its O and LSE device->host.  Two device
    # buffer sets and a copy stream let step i+1's inputs and step i-1's results move while
    # step i computes, as a serving loop would.  The pipeline's ends are cut into KV-head groups
    # (the query heads of one KV head and that KV head): the first step computes each group as
    # soon as its inputs have landed, and the last step sends each group's O and LSE back as soon
    # as it is computed, so only one group's upload and one group's download stay exposed.
    e2e = None
    if rank == 0 or world > 1:
        hq_, hk_, hv_ = (t.cpu().pin_memory() for t in (q, k, v))
        ho = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        bufs = [tuple(torch.empty_like(t) for t in (q, k, v, out, lse)) for _ in range(2)]
        copy = torch.cuda.Stream(dev)
        n_e2e = max(3, min(args.steps, 20))
        group = w.Hq // w.Hkv
        # KV-head groups (a few of them: enough to shorten the exposed ends, few launches); with
        # B > 1 a head slice is not contiguous, and the LSE output must be, so one group
        n_groups = max(g for g in (1, 2, 4, 8) if w.Hkv % g == 0) if w.B == 1 else 1
        kv_per = w.Hkv // n_groups
        heads = [(gi * kv_per * group, (gi + 1) * kv_per * group, gi * kv_per, (gi + 1) * kv_per)
                 for gi in range(n_groups)]
        loaded = [torch.cuda.Event() for _ in range(n_e2e)]
        computed = [torch.cuda.Event() for _ in range(n_e2e)]
        drained = [torch.cuda.Event() for _ in range(n_e2e)]
        part_loaded = [torch.cuda.Event() for _ in range(n_groups)]
        part_computed = [torch.cuda.Event() for _ in range(n_groups)]

        def h2d(i):
            dq, dk, dv = bufs[i % 2][:3]
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(computed[i - 2])  # the buffer set is free again
                if i == 0:
                    for gi, (h0, h1, g0, g1) in enumerate(heads):
                        dq[:, h0:h1].copy_(hq_[:, h0:h1], non_blocking=True)
                        dk[:, g0:g1].copy_(hk_[:, g0:g1], non_blocking=True)
                        dv[:, g0:g1].copy_(hv_[:, g0:g1], non_blocking=True)
                        part_loaded[gi].record(copy)
                else:
                    dq.copy_(hq_, non_blocking=True)
                    dk.copy_(hk_, non_blocking=True)
                    dv.copy_(hv_, non_blocking=True)
                loaded[i].record(copy)

        def e2e_run(n):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            start.record(stream)
            copy.wait_stream(stream)
            h2d(0)
            for i in range(n):
                if i + 1 < n:
                    h2d(i + 1)
                dq, dk, dv, do, dl = bufs[i % 2]
                by_group = i == 0 or i == n - 1
                with torch.cuda.stream(stream):
                    if not by_group:
                        stream.wait_event(loaded[i])
                        attn.attn_fwd(dq, dk, dv, causal=w.causal, sm_scale=w.sm_scale, out=do,
                                      lse=dl)
                    else:
                        if i > 0:
                            stream.wait_event(loaded[i])
                        for gi, (h0, h1, g0, g1) in enumerate(heads):
                            if i == 0:
                                stream.wait_event(part_loaded[gi])
                            attn.attn_fwd(dq[:, h0:h1], dk[:, g0:g1], dv[:, g0:g1],
                                          causal=w.causal, sm_scale=w.sm_scale,
                                          out=do[:, h0:h1], lse=dl[:, h0:h1])
                            part_computed[gi].record(stream)
                    computed[i].record(stream)
                with torch.cuda.stream(copy):
                    if i == n - 1:
                        for gi, (h0, h1, _, _) in enumerate(heads):
                            copy.wait_event(part_computed[gi])
                            ho[i % 2][:, h0:h1].copy_(do[:, h0:h1], non_blocking=True)
                            hl[i % 2][:, h0:h1].copy_(dl[:, h0:h1], non_blocking=True)
                    else:
                        copy.wait_event(computed[i])
                        ho[i % 2].copy_(do, non_blocking=True)
                        hl[i % 2].copy_(dl, non_blocking=True)
                    drained[i].record(copy)
            stream.wait_event(drained[n - 1])
            end.record(stream)
            torch.cuda.synchronize()
            return start.elapsed_time(end)

        e2e_run(2)
        # the host<->device copy rate can vary from run to run (the host's memory system may be
        # busy with other work): three runs, the median one reported, all three listed
        runs = sorted(e2e_run(n_e2e) for _ in range(3))
        total = runs[1]
        # the last step's results, back on the host, match the device-side run's (the grouped
        # launches compute the same heads; a group small enough to be split differs by rounding)
        d_o = (ho[(n_e2e - 1) % 2].float() - out.cpu().float()).abs().max().item()
        d_l = (hl[(n_e2e - 1) % 2] - lse.cpu()).abs().max().item()
        if not (d_o <= 2e-2 and d_l <= 1e-3):
            raise SystemExit(f"end-to-end results differ from the device-side run ({d_o}, {d_l})")
        h2d_b = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
        d2h_b = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
        e2e = {"value": w.flops * n_e2e / (total * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
               "ms_per_step": total / n_e2e, "steps": n_e2e,
               "runs_ms_per_step": [r / n_e2e for r in runs], "reported": "median of 3 runs",
               "overlap": (f"copies of neighbouring steps overlap compute (2 buffer sets); the "
                           f"first step's upload and the last step's download move in "
                           f"{n_groups} KV-head groups, each group computed as its inputs land "
                           f"and sent back as it is computed")}

    # ---- context: the other long-context lengths (same kernel), not the headline -------------
    sweep = []
    gpu_out = {}  # CPU copies of GPU outputs the CPU-baseline leg compares with the oracle

    def keep_rows(wk, o, l):  # the rows the parity tests sample, for the long lengths
        rows = wl.sample_rows(wk, 64).long()
        oc, lc = o.cpu(), l.cpu()
        gpu_out[wk.name] = (
            torch.stack([oc[b, h][rows[b, h]] for b in range(wk.B) for h in range(wk.Hq)])
            .reshape(wk.B, wk.Hq, -1, wk.D),
            torch.stack([lc[b, h][rows[b, h]] for b in range(wk.B) for h in range(wk.Hq)])
            .reshape(wk.B, wk.Hq, -1))

    if not args.no_sweep and rank == 0:
        for n in sorted(wl.LONG):
            if n == w.N and w.name.startswith("long"):
                sweep.append({"N": n, "ms": mean_launch_ms, "tflops": achieved,
                              "frac": achieved / peak})
                keep_rows(w, out, lse)
                continue
            ws = wl.LONG[n]
            sq, sk, sv = (t.to(dev) for t in wl.make_qkv(ws))
            so, sl = torch.empty_like(sq), torch.empty(ws.B, ws.Hq, ws.N, dtype=torch.float32,
                                                       device=dev)

            def sstep():
                attn.attn_fwd(sq, sk, sv, causal=ws.causal, sm_scale=ws.sm_scale, out=so, lse=sl)

            with torch.cuda.stream(stream):
                for _ in range(3):
                    sstep()
            ms = statistics.mean(timed_launches(sstep, stream, 20))
            tf = ws.flops / (ms * 1e-3) / 1e12
            sweep.append({"N": n, "ms": ms, "tflops": tf, "frac": tf / peak})
            keep_rows(ws, so, sl)
            del sq, sk, sv, so, sl

    # ---- context: the two D = 128 forward kernels side by side (the one-CTA kernel attn_fwd
    # runs, and the CTA-pair kernel whose M = 256 MMAs span two SMs), through the test hook -----
    kernels = []
    if not args.no_sweep and rank == 0:
        lib = _lib.load()
        sh = ctypes.c_void_p(stream.cuda_stream)
        for wk in (wl.LONG[8192], wl.LONG[32768]):
            kq, kk_, kv_ = (t.to(dev) for t in wl.make_qkv(wk))
            ko = torch.empty_like(kq)
            kl = torch.empty(wk.B, wk.Hq, wk.N, dtype=torch.float32, device=dev)
            kargs = (kq.data_ptr(), kk_.data_ptr(), kv_.data_ptr(), ko.data_ptr(), kl.data_ptr(),
                     wk.B, wk.Hq, wk.Hkv, wk.N, wk.D, int(wk.causal), ctypes.c_float(wk.sm_scale))
            entry = {"workload": wk.name}
            for name, kid in (("one_cta", 1), ("pair", 2)):
                def kstep(kid=kid):
                    assert lib.attn_fwd_test_kernel(*kargs, kid, -1, sh) == 0

                with torch.cuda.stream(stream):
                    for _ in range(3):
                        kstep()
                ms = statistics.median(timed_launches(kstep, stream, 10))
                entry[f"{name}_ms"] = ms
                entry[f"{name}_tflops"] = wk.flops / (ms * 1e-3) / 1e12
            kernels.append(entry)
            del kq, kk_, kv_, ko, kl
        if attn.device_status(dev) != 0:
            raise SystemExit("device status word reports an expired wait in the kernels leg")

    # ---- context: wide heads (D = 256, one Q tile per CTA) on a long causal sequence ---------
    wide = []
    if not args.no_sweep and rank == 0:
        ww = wl.WIDE
        wq, wk, wv = (t.to(dev) for t in wl.make_qkv(ww))
        wo = torch.empty_like(wq)
        wlse = torch.empty(ww.B, ww.Hq, ww.N, dtype=torch.float32, device=dev)

        def wstep():
            attn.attn_fwd(wq, wk, wv, causal=ww.causal, sm_scale=ww.sm_scale, out=wo, lse=wlse)

        with torch.cuda.stream(stream):
            for _ in range(3):
                wstep()
        ms = statistics.median(timed_launches(wstep, stream, 20))
        tf = ww.flops / (ms * 1e-3) / 1e12
        wide.append({"workload": ww.name, "ms": ms, "tflops": tf, "frac": tf / peak})
        del wq, wk, wv, wo, wlse

    # ---- context: the five configurations (single pass, C-ABI, cold L2) ------------------------
    # ms, TFLOPS against the tensor peak and algorithmic GB/s against the copy bandwidth: the short
    # sequences are bound by latency and occupancy rather than by either roofline.
    configs = []
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if not args.no_sweep else None
    if not args.no_sweep and rank == 0:
        hbm = float(peaks["hbm_gbs"])
        lib = _lib.load()
        sh = ctypes.c_void_p(stream.cuda_stream)
        for wc in (wl.TINY_NONCAUSAL, wl.TINY_CAUSAL, wl.GQA4_CAUSAL, wl.GQA8_CAUSAL, wl.MHA,
                   wl.MHA_OUTLIER, wl.MQA):
            cq, ck, cv = (t.to(dev) for t in wl.make_qkv(wc))
            co = torch.empty_like(cq)
            cl = torch.empty(wc.B, wc.Hq, wc.N, dtype=torch.float32, device=dev)
            cargs = (cq.data_ptr(), ck.data_ptr(), cv.data_ptr(), co.data_ptr(), cl.data_ptr(),
                     wc.B, wc.Hq, wc.Hkv, wc.N, wc.D, int(wc.causal), ctypes.c_float(wc.sm_scale),
                     sh)

            def cstep():
                assert lib.attn_fwd(*cargs) == 0

            ms = cold_launch_ms(cstep, stream, flush, 20)
            tf = wc.flops / (ms * 1e-3) / 1e12
            gbs = wc.bytes / (ms * 1e-3) / 1e9
            configs.append({"workload": wc.name, "B": wc.B, "Hq": wc.Hq, "Hkv": wc.Hkv, "N": wc.N,
                            "D": wc.D, "causal": wc.causal, "us": ms * 1e3, "tflops": tf,
                            "frac": tf / peak, "gbs": gbs, "hbm_frac": gbs / hbm,
                            "l2": "256 MB flush before each launch"})
            gpu_out[wc.name] = (co.cpu(), cl.cpu())
            del cq, ck, cv, co, cl

    # ---- context: low-occupancy configurations: attn_fwd (which may split the key axis into
    # clusters itself), the forced single pass and the split-KV entry point ---------------------
    low_occ = []
    if not args.no_sweep and rank == 0:
        for ws_ in (wl.MHA, wl.MQA, wl.FEWHEADS, wl.FEWHEADS_CAUSAL):
            lq, lk, lv = (t.to(dev) for t in wl.make_qkv(ws_))
            lo = torch.empty_like(lq)
            ll = torch.empty(ws_.B, ws_.Hq, ws_.N, dtype=torch.float32, device=dev)
            # split-KV: the library's default, or 2 forced splits where it declines to split
            dflt = attn.splitkv_num_splits(ws_.B, ws_.Hq, ws_.N, ws_.D, ws_.causal)
            n_sp = max(2, dflt)
            wbuf = torch.empty(max(1, attn.splitkv_workspace_bytes(ws_.B, ws_.Hq, ws_.N, ws_.D,
                                                                   n_sp)),
                               dtype=torch.uint8, device=dev)

            # Pre-bound C-ABI calls: these kernels take ~15-100 us, not much more than the Python
            # binding's per-call host time, which would otherwise be what gets measured.
            lib = _lib.load()
            sh = ctypes.c_void_p(stream.cuda_stream)
            common = (lq.data_ptr(), lk.data_ptr(), lv.data_ptr(), lo.data_ptr(), ll.data_ptr(),
                      ws_.B, ws_.Hq, ws_.Hkv, ws_.N, ws_.D, int(ws_.causal),
                      ctypes.c_float(ws_.sm_scale))

            def fwd():
                assert lib.attn_fwd(*common, sh) == 0

            def single():  # one split: the single pass, never split further
                assert lib.attn_fwd_splitkv(*common, 1, None, 0, sh) == 0

            def split():
                assert lib.attn_fwd_splitkv(*common, n_sp, wbuf.data_ptr(), wbuf.numel(), sh) == 0

            entry = {"workload": ws_.name, "causal": ws_.causal,
                     "attn_fwd_splits": attn.fwd_num_splits(ws_.B, ws_.Hq, ws_.N, ws_.D,
                                                            ws_.causal),
                     "splits": n_sp, "library_choice": dflt}
            for name, fn in (("attn_fwd", fwd), ("single", single), ("splitkv", split)):
                ms = cold_launch_ms(fn, stream, flush, 30)
                entry[f"{name}_us"] = ms * 1e3
                entry[f"{name}_tflops"] = ws_.flops / (ms * 1e-3) / 1e12
                entry[f"{name}_gbs"] = ws_.bytes / (ms * 1e-3) / 1e9
            low_occ.append(entry)
            del lq, lk, lv, lo, ll, wbuf

    # ---- context: the backward (by recompute) on the long-context workload -------------------
    # Algorithmic FLOPs of the backward: 2.5x the forward's (five N x N x D matmuls: S, dP, dV,
    # dK, dQ), halved under the causal mask like the forward's.
    backward = []
    if not args.no_sweep and rank == 0:
        for n in (8192, 16384):
            wb = wl.LONG[n]
            bq, bk, bv = (t.to(dev) for t in wl.make_qkv(wb))
            bo, bl = attn.attn_fwd(bq, bk, bv, causal=wb.causal, sm_scale=wb.sm_scale)
            g = torch.Generator(device="cpu").manual_seed(77)
            bdo = torch.randn(bq.shape, generator=g).to(torch.bfloat16).to(dev)
            dq, dk, dv = torch.empty_like(bq), torch.empty_like(bk), torch.empty_like(bv)
            lib = _lib.load()
            need = int(lib.attn_bwd_workspace_bytes(wb.B, wb.Hq, wb.N))
            wsb = torch.empty(need, dtype=torch.uint8, device=dev)
            sh = ctypes.c_void_p(stream.cuda_stream)

            def bstep():
                assert lib.attn_bwd(bq.data_ptr(), bk.data_ptr(), bv.data_ptr(), bo.data_ptr(),
                                    bl.data_ptr(), bdo.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), wb.B, wb.Hq, wb.Hkv, wb.N, wb.D,
                                    int(wb.causal), ctypes.c_float(wb.sm_scale), wsb.data_ptr(),
                                    need, sh) == 0

            with torch.cuda.stream(stream):
                for _ in range(3):
                    bstep()
            ms = statistics.median(timed_launches(bstep, stream, 10))
            tf = 2.5 * wb.flops / (ms * 1e-3) / 1e12
            backward.append({"workload": wb.name, "ms": ms, "tflops": tf, "frac": tf / peak,
                             "kernels_per_step": 3})
            del bq, bk, bv, bo, bl, bdo, dq, dk, dv, wsb
        if attn.device_status(dev) != 0:
            raise SystemExit("device status word reports an expired wait in the backward leg")

    # ---- context: absorbed MLA decode (the second workload), one decode query per head --------
    # HBM-bound at large batch: reported as GB/s of algorithmic bytes (cache + queries read once,
    # out_c and LSE written) against the measured copy bandwidth.  The 256 MB flush before each
    # launch keeps the cache out of L2 for the small batches.
    mla = []
    if not args.no_sweep and rank == 0:
        hbm = float(peaks["hbm_gbs"])
        lib = _lib.load()
        sh = ctypes.c_void_p(stream.cuda_stream)
        for wm in (wl.MLA_B1[4096], wl.MLA_B1[16384], wl.MLA_B32):
            mq, mkv = wl.make_mla(wm, device=dev)
            mo = torch.empty(wm.B, wm.H, attn.MLA_D_C, dtype=torch.bfloat16, device=dev)
            ml = torch.empty(wm.B, wm.H, dtype=torch.float32, device=dev)
            n_sp = attn.mla_decode_num_splits(wm.B, wm.H, wm.T)
            need = attn.mla_decode_workspace_bytes(wm.B, wm.H, wm.T, n_sp)
            mws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            args_ = (mq.data_ptr(), mkv.data_ptr(), mo.data_ptr(), ml.data_ptr(), wm.B, wm.H, wm.T,
                     attn.MLA_D_C, attn.MLA_D_R, ctypes.c_float(wm.sm_scale), n_sp,
                     mws.data_ptr(), need)

            def mstep():
                assert lib.attn_mla_decode(*args_, sh) == 0

            ms = cold_launch_ms(mstep, stream, flush, 20, warm=5)
            gbs = wm.bytes / (ms * 1e-3) / 1e9
            mla.append({"workload": wm.name, "us": ms * 1e3, "gbs": gbs, "hbm_frac": gbs / hbm,
                        "tflops": wm.flops / (ms * 1e-3) / 1e12, "splits": n_sp,
                        "kernels_per_step": 2 if n_sp > 1 else 1})
            del mq, mkv, mo, ml, mws
        if attn.device_status(dev) != 0:
            raise SystemExit("device status word reports an expired wait in the MLA leg")

    # ---- CPU baseline: the oracle as it stands, bounded sample, rank 0 at N=1 only -----------
    cpu = None
    cpu_table = []
    if rank == 0 and world == 1:
        import oracle

        qc, kc, vc = (t.cpu() for t in (q, k, v))
        n_rows, _ = time_oracle(w, qc, kc, vc, args.cpu_seconds)
        rows = cpu_sample_rows(w, n_rows)
        t0 = time.perf_counter()
        oracle.attn_ref(qc, kc, vc, w.causal, w.sm_scale, rows=rows.numpy())
        dt = time.perf_counter() - t0
        f = sample_flops(w, rows)
        cpu = {"value": f / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(),
               "kind": "oracle",
               "sample": f"{n_rows} seeded query rows per head x {w.B * w.Hq} heads of {w.name}; "
                         f"{f / 1e9:.2f} GFLOP in {dt:.1f} s"}
        if not args.no_sweep:
            gpu_us = {c["workload"]: c["us"] for c in configs}
            gpu_us.update({f"long-gqa8-causal-n{x['N']}": x["ms"] * 1e3 for x in sweep})
            cpu_table = cpu_baseline_table(gpu_us, gpu_out)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, "inputs and output exceed the 129 MB L2; no flush"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clocks, "configs": configs, "sweep": sweep,
            "low_occupancy": low_occ, "wide_heads": wide, "forward_kernels": kernels,
            "backward": backward,
            "mla_decode": mla, "cpu_baseline_table": cpu_table,
            "kernel_sha": kernel_hash(),
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
