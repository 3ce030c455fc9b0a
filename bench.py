"""Benchmark of channels-last GroupNorm+SiLU on GB300 (one JSON line on stdout).

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                    [--workload NAME] [--variant auto|fused|two_pass] [--no-sweep]

A step is one call of the whole path (pass 1, finalize, pass 2) on one
synthetic bf16 activation of the workload (default: N=1 C=256 H=W=1024, the
FLUX.2 VAE up-block GroupNorm shape, 512 MiB: the largest configuration).
Inputs are seeded (see
``channels_last_groupnorm_gb300/workloads.py``) and already resident in HBM;
consecutive steps rotate over enough buffer sets that no step finds its
input in L2.  The timed steps are captured once into a CUDA graph and
replayed (``--launch stream`` launches them one by one instead).  ``value``
is effective bandwidth: N*L*C*4 bytes (read x once,
write y once) per step, summed over ranks, divided by the slowest rank's
time.  ``e2e`` repeats the measurement through the C ABI from pinned host
buffers with the host<->device copies inside the timed region.

``--workload upconv_*`` measures the fused nearest-2x upsample + 3x3 conv
of the decoder's up-samplers instead (TFLOP/s against the measured bf16
tensor peak), ``--workload attn_*`` the mid-block attention with the output
projection folded into V, ``--workload rga_*`` the residual-gate update;
the default run adds all three to its sweep.

Under torchrun each rank runs its own replica on its own GPU (the
operation has no cross-GPU exchange); rank 0 prints the line.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
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

METRIC = "NHWC GroupNorm+SiLU µs/call and HBM GB/s (% of GB300 peak), bf16 G=32"
DEFAULT_WORKLOAD = "gn_silu_c256_1024x1024"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
UPCONV_METRIC = "fused nearest-2x upsample + 3x3 conv, bf16 in/out, fp32 accumulate: us/call and TFLOP/s"
ATTN_METRIC = ("single-head attention, output projection folded into V, bf16 in/out, fp32 scores and "
               "accumulation: us/call and TFLOP/s")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
KERNEL_SOURCES = ["gn_kernels.cu", "gn_cluster.cu", "gn_capi.cu", "gn_internal.h", "gn_math.cuh", "gn_ptx.cuh",
                  "capi_util.h", "rga_kernels.cu"]
# the files that make the upsample-conv kernels and their launch plan (the
# C-ABI checks in tc_capi.cu do not change what runs on the GPU)
UPCONV_SOURCES = ["upconv_kernels.cu", "tc_ptx.cuh", "tc_common.cuh", "gn_ptx.cuh"]
ATTN_SOURCES = ["attn_kernels.cu", "tc_ptx.cuh", "tc_common.cuh", "tc_internal.h", "tc_capi.cu", "gn_ptx.cuh"]


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; also exercised with gloo on CPU by the tests)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_timing(elapsed_s: float, units: float, device=None):
    """(max elapsed over ranks, sum of units over ranks); identity when not
    distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# peaks, clocks, traffic
# ---------------------------------------------------------------------------
def tensor_peak():
    """Measured dense bf16 TFLOP/s (cuBLAS burst) of the GB300s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "of measured (burst)", float(d.get("bf16_tflops_sustained", 0)) or None
    except (OSError, ValueError, KeyError):
        return FALLBACK_BF16_TFLOPS, "of fallback", None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "of measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "of fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("", "[N/A]") else None,
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons),
                "power_w_max": max((r["power"] for r in rows if r["power"] is not None),
                                   default=None)}


def kernel_source_hash(sources=None) -> str:
    """Hash of the code of the given source files, with comments and
    blank lines removed: an edit of comments leaves recorded counters valid."""
    import re
    h = hashlib.sha256()
    for name in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, "channels_last_groupnorm_gb300", "csrc", name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"(^|\s)//.*$", r"\1", text, flags=re.M)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, variant: str, sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    src = kernel_source_hash(sources)
    for line in lines:
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#"):
            wname, var, sha, nbytes = parts
            if wname == workload and var == variant and sha == src:
                return float(nbytes)
    return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def upload(case, device):
    import numpy as np
    import torch
    x = torch.from_numpy(case["x_bits"].view(np.int16)).to(device).view(torch.bfloat16)
    return (x.contiguous(), torch.from_numpy(case["gamma"]).to(device),
            torch.from_numpy(case["beta"]).to(device))


def buffer_sets_for(nbytes_per_set: int, l2_bytes: int, cap: int = 64) -> int:
    """Enough rotating buffer sets that the sets together exceed twice L2."""
    need = -(-2 * l2_bytes // max(1, nbytes_per_set))
    return int(max(1, min(cap, need)))


def time_calls(call, nsets, steps, stream):
    """Per-step CUDA-event durations (ms) of `steps` calls rotating over the
    buffer sets, plus the total elapsed time of the region (s)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        call(i % nsets)
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, t0.elapsed_time(t1) / 1e3


def capture_steps(call, nsets, steps, stream):
    """A CUDA graph holding `steps` consecutive calls (rotating over the
    buffer sets), or None if the calls cannot be captured."""
    import torch
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                call(i % nsets)
    except Exception:   # noqa: BLE001 -- any capture failure falls back to stream launches
        torch.cuda.synchronize()
        return None
    return graph


def time_graph(graph, stream):
    """Elapsed time (s) of one replay of a captured sequence of steps."""
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return t0.elapsed_time(t1) / 1e3


def raw_entry(w):
    """The C entry point a workload goes through: gn_silu_rows_any for a C
    that is not a power of two (and for 5D input), else gn_silu_rows_ex."""
    from channels_last_groupnorm_gb300 import gnsilu as gs
    return gs.raw_gn_silu_rows_any if (w.general or w.D > 1) else gs.raw_gn_silu_rows_ex


def line_config(w, silu, world):
    """The `config` of a GroupNorm line; both arms print the same one."""
    return {**w.describe(), "silu": bool(silu),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (rotating buffer sets of x + y that together exceed twice L2)",
            "bytes_per_step": "N*L*C*4 (x read once, y written once)"}


def measure_workload(w, variant_id, steps, warmup, device, stream, soak_s=0.0, sampler=None,
                     seeded=True, launch="graph", hot_l2=False, apply_silu=True):
    """Device-resident timing of one workload.  Returns a dict."""
    import torch
    from channels_last_groupnorm_gb300 import gnsilu as gs
    from channels_last_groupnorm_gb300 import workloads as wl

    if seeded:
        x0, gamma, beta = upload(wl.make_inputs(w), device)
    else:   # same distributions drawn on the device (sweep of the larger shapes)
        gen = torch.Generator(device=device).manual_seed(1000 + w.index)
        x0 = (torch.randn(w.N, w.L, w.C, generator=gen, device=device) * w.x_std
              + w.x_mean).to(torch.bfloat16)
        gamma_np, beta_np = wl.affine_params(w.index, w.C)
        gamma = torch.from_numpy(gamma_np).to(device)
        beta = torch.from_numpy(beta_np).to(device)
    elems = w.elements
    set_bytes = 4 * elems
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = 1 if hot_l2 else buffer_sets_for(set_bytes, l2)
    free, _ = torch.cuda.mem_get_info(device)
    nsets = max(1, min(nsets, int(0.5 * free // set_bytes)))
    xs = [x0] + [x0.clone() for _ in range(nsets - 1)]
    ys = [torch.empty_like(x0) for _ in range(nsets)]
    h = stream.cuda_stream
    entry = raw_entry(w)
    silu = 1 if apply_silu else 0

    def call(i):
        rc = entry(xs[i].data_ptr(), gamma.data_ptr(), beta.data_ptr(), ys[i].data_ptr(), w.N, w.L,
                   w.C, w.G, w.eps, silu, variant=variant_id, stream=h)
        if rc != 0:
            raise RuntimeError(f"{entry.__name__} failed: {gs.status_string(rc)}")

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            call(i % nsets)
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.start()
        if soak_s > 0:
            t_end = time.time() + soak_s
            i = 0
            while time.time() < t_end:
                for _ in range(50):
                    call(i % nsets)
                    i += 1
                torch.cuda.synchronize()
        before = gs.gn_kernel_launch_count()
        call(0)
        per_call = gs.gn_kernel_launch_count() - before   # kernels one call launches
        graph = capture_steps(call, nsets, steps, stream) if launch == "graph" else None
        if graph is not None:
            graph.replay()                      # upload + warm the graph
            elapsed = time_graph(graph, stream)
            per = [elapsed * 1e3 / steps] * steps
            mode = "cuda-graph"
        else:
            per, elapsed = time_calls(call, nsets, steps, stream)
            mode = "stream"
        launches = per_call * steps
        clocks = sampler.stop() if sampler is not None else None
        del graph
    status = gs.gn_device_status(False)
    if status != 0:
        raise RuntimeError(f"device status after timing: {gs.status_string(status)}")
    res = {"elapsed_s": elapsed, "per_step_ms": per, "nsets": nsets, "set_bytes": set_bytes,
           "launches": launches, "clocks": clocks, "launch": mode,
           "variant": {1: "two_pass", 2: "fused", 3: "cluster"}.get(
               gs.gn_silu_pick_variant(w.N, w.L, w.C, w.G) if variant_id == 0 else variant_id,
               "?")}
    del xs, ys
    torch.cuda.empty_cache()
    return res


def measure_e2e(w, variant_id, steps, warmup, device, stream):
    """Through the C ABI from pinned host buffers: every step copies x,
    gamma and beta in, makes the call and copies y out, all inside the timed
    region.  The steps are pipelined the way a streaming caller runs them:
    copies in and out go on two copy streams with two device buffer sets,
    so step i's call overlaps step i+1's copy in and step i-1's copy out;
    the region runs from the first copy in to the last copy out."""
    import numpy as np
    import torch
    from channels_last_groupnorm_gb300 import gnsilu as gs
    from channels_last_groupnorm_gb300 import workloads as wl

    case = wl.make_inputs(w)
    hx = torch.from_numpy(case["x_bits"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hg = torch.from_numpy(case["gamma"]).pin_memory()
    hb = torch.from_numpy(case["beta"]).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    dx = [torch.empty_like(hx, device=device) for _ in range(2)]
    dg = [torch.empty_like(hg, device=device) for _ in range(2)]
    db = [torch.empty_like(hb, device=device) for _ in range(2)]
    dy = [torch.empty_like(hx, device=device) for _ in range(2)]
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    h = stream.cuda_stream
    entry = raw_entry(w)

    def run(n, timed):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_k = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if timed:
            barrier()
            torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_k[i - 2])      # the call two steps back has read this set
                dx[k].copy_(hx, non_blocking=True)
                dg[k].copy_(hg, non_blocking=True)
                db[k].copy_(hb, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])      # y of two steps back has left the device
            rc = entry(dx[k].data_ptr(), dg[k].data_ptr(), db[k].data_ptr(), dy[k].data_ptr(),
                       w.N, w.L, w.C, w.G, w.eps, 1, variant=variant_id, stream=h)
            if rc != 0:
                raise RuntimeError(gs.status_string(rc))
            ev_k[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[i])
                hy.copy_(dy[k], non_blocking=True)
                ev_out[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        if timed:
            barrier()
        return t0.elapsed_time(t1) / 1e3

    run(max(3, warmup), False)
    elapsed = run(steps, True)
    h2d = hx.numel() * 2 + hg.numel() * 4 + hb.numel() * 4
    d2h = hy.numel() * 2
    return elapsed, h2d, d2h


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or ''."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


_ORACLE_CORES = None


def oracle_cores(orc) -> int:
    """The oracle's OpenMP thread count before anything set it to one
    thread (a one-thread run changes the process-wide default)."""
    global _ORACLE_CORES
    if _ORACLE_CORES is None:
        _ORACLE_CORES = orc.max_threads()
    return _ORACLE_CORES


def time_oracle(orc, case, w, silu, budget_s, max_calls, nthreads=0):
    """Mean seconds per full oracle call, over calls until `budget_s` has
    passed (at least one, at most `max_calls`)."""
    t0 = time.perf_counter()
    calls = 0
    while True:
        orc.forward(case["x_bits"], case["gamma"], case["beta"], w.G, w.eps, silu, nthreads=nthreads)
        calls += 1
        if time.perf_counter() - t0 >= budget_s or calls >= max_calls:
            break
    return (time.perf_counter() - t0) / calls, calls


def cpu_baseline(w, budget_s=10.0, case=None):
    """The fp64 oracle on this host's cores, on the full workload tensor,
    repeated until about `budget_s` of CPU time has passed; plus a
    single-thread run."""
    import oracle
    from channels_last_groupnorm_gb300 import workloads as wl
    case = case or wl.make_inputs(w)
    orc = oracle.get()
    cores = oracle_cores(orc)
    dt, calls = time_oracle(orc, case, w, True, budget_s, 50, nthreads=cores)
    dt1, calls1 = time_oracle(orc, case, w, True, budget_s / 4, 20, nthreads=1)
    return {"value": round(4.0 * w.elements / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "us_per_call": round(dt * 1e6, 1), "cpu_model": cpu_model(),
            "one_thread": {"value": round(4.0 * w.elements / dt1 / 1e9, 4), "unit": "GB/s",
                           "us_per_call": round(dt1 * 1e6, 1), "calls": calls1},
            "sample": f"{calls} full calls of the fp64 oracle on the {w.name} tensor "
                      f"({w.elements} elements), {cores} OpenMP threads; {calls1} on one thread"}


def cpu_baselines(budget_s=1.0):
    """The fp64 oracle on every configuration (and both SiLU settings of the
    one run with and without it), all host cores and one thread: one full
    call or more each, µs/call and GB/s at 4 B/elem."""
    import oracle
    from channels_last_groupnorm_gb300 import workloads as wl
    orc = oracle.get()
    cores = oracle_cores(orc)
    out = []
    for w in wl.WORKLOADS:
        case = wl.make_inputs(w)
        for silu in w.silu_modes:
            dt, _ = time_oracle(orc, case, w, silu, budget_s, 20, nthreads=cores)
            dt1, _ = time_oracle(orc, case, w, silu, budget_s / 2, 5, nthreads=1)
            out.append({"workload": w.name, "silu": silu, "cores": cores,
                        "us": round(dt * 1e6, 1), "gbs": round(4.0 * w.elements / dt / 1e9, 3),
                        "us_1t": round(dt1 * 1e6, 1), "gbs_1t": round(4.0 * w.elements / dt1 / 1e9, 3)})
        del case
    return out


def sweep(variant_id, device, stream, peak, launch="graph"):
    """Every workload shape (and SiLU setting), the general-channel ones
    included: us/call and effective bandwidth at 4 B/elem (read once + write
    once) and 6 B/elem (two-pass byte count)."""
    from channels_last_groupnorm_gb300 import workloads as wl
    out = []
    for w in wl.WORKLOADS + wl.GENERAL_WORKLOADS:
        for silu in w.silu_modes:
            r = measure_workload(w, variant_id, 30, 5, device, stream, seeded=(w.elements <= 1 << 24),
                                 launch=launch, apply_silu=silu)
            us = statistics.median(r["per_step_ms"]) * 1e3
            gbs4 = 4.0 * w.elements / (us * 1e-6) / 1e9
            gbs6 = 6.0 * w.elements / (us * 1e-6) / 1e9
            hot = None
            if w.elements <= 1 << 25:
                # the small shapes also with one buffer set: x and y stay in L2
                rh = measure_workload(w, variant_id, 30, 5, device, stream, seeded=(w.elements <= 1 << 24),
                                      launch=launch, hot_l2=True, apply_silu=silu)
                hot = round(statistics.median(rh["per_step_ms"]) * 1e3, 2)
            out.append({"workload": w.name, "C": w.C, "silu": silu, "variant": r["variant"],
                        "us_per_call": round(us, 2), "us_per_call_hot_l2": hot,
                        "gbs_4B": round(gbs4, 1), "gbs_6B": round(gbs6, 1),
                        "frac_4B": round(gbs4 / peak, 3), "frac_6B": round(gbs6 / peak, 3),
                        "pages_h200_us": w.pages_us_h200,
                        "l2": f"{r['nsets']} rotating buffer sets of {r['set_bytes'] >> 20} MiB",
                        "launch": r["launch"]})
    return out


def compact_sweep(rows):
    """One short string per swept shape, so the figures survive a reader
    that keeps only the end of the line."""
    out = []
    for r in rows:
        name = r["workload"].replace("gn_silu_", "").replace("gn_", "")
        out.append(f"{name}{'' if r['silu'] else ' nosilu'} {r['variant']} {r['us_per_call']}us "
                   f"4B={r['frac_4B']} 6B={r['frac_6B']}"
                   + (f" hotL2={r['us_per_call_hot_l2']}us" if r["us_per_call_hot_l2"] else "")
                   + (f" h200={r['pages_h200_us']}us" if r["pages_h200_us"] else ""))
    return out


def measure_rga(w, fmt, steps, device, stream, peak):
    """gn_residual_gate_add on one residual-gate workload: CUDA-graph
    replay of `steps` calls over rotating buffer sets (together more than
    twice L2), µs per call and GB/s at 6 B per element (residual and update
    read, y written; the gate row is negligible)."""
    import torch
    from channels_last_groupnorm_gb300 import gnsilu as gs
    from channels_last_groupnorm_gb300 import workloads as wl
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[fmt]
    r0, u0, g0 = (t.to(dt).to(device) for t in wl.make_rga_inputs(w))
    set_bytes = 6 * w.elements
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = buffer_sets_for(set_bytes, l2)
    sets = [(r0.clone(), u0.clone(), torch.empty_like(r0)) for _ in range(nsets)]
    h = stream.cuda_stream
    code = {"bf16": 0, "fp16": 1}[fmt]

    def call(i):
        r, u, y = sets[i]
        rc = gs.raw_gn_residual_gate_add(r.data_ptr(), u.data_ptr(), g0.data_ptr(), y.data_ptr(), w.rows, w.D,
                                         code, stream=h)
        if rc != 0:
            raise RuntimeError(gs.status_string(rc))

    with torch.cuda.stream(stream):
        for i in range(5):
            call(i % nsets)
        torch.cuda.synchronize()
        graph = capture_steps(call, nsets, steps, stream)
        graph.replay()
        elapsed = time_graph(graph, stream)
        del graph
    us = elapsed * 1e6 / steps
    gbs = 6.0 * w.elements / (us * 1e-6) / 1e9
    del sets
    torch.cuda.empty_cache()
    return {"workload": w.name, "format": fmt, "us_per_call": round(us, 2), "gbs_6B": round(gbs, 1),
            "frac_6B": round(gbs / peak, 3), "pages_fused_us_h200": w.pages_us_h200,
            "pages_eager_us_h200": w.pages_eager_us_h200,
            "l2": f"{nsets} rotating buffer sets of {set_bytes >> 20} MiB", "launch": "cuda-graph"}


def upconv_device_inputs(w, device):
    import numpy as np
    import torch
    from channels_last_groupnorm_gb300 import workloads as wl
    c = wl.make_upconv_inputs(w)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)
    x = dev(c["x_bits"]).reshape(w.N, w.H, w.W, w.Cin)
    wt = dev(c["w_bits"]).reshape(w.Cout, w.Cin, 3, 3).contiguous()
    b = dev(c["bias_bits"]) if c["bias_bits"] is not None else None
    return c, x, wt, b


def measure_upconv(w, steps, device, stream, peak, cudnn_context=True):
    """gn_upconv_nhwc on one decoder up-sampler workload: the weight is
    folded once (gn_upconv_fold, untimed: it is per model, not per call),
    then a CUDA graph of `steps` calls is replayed over rotating (x, y)
    sets that together exceed twice L2.  TFLOP/s counts the folded
    evaluation's multiply-adds (2 x 4 Cin per output element)."""
    import torch
    import torch.nn.functional as F
    from channels_last_groupnorm_gb300 import gnsilu as gs
    _, x0, wt, b = upconv_device_inputs(w, device)
    wf = gs.upconv_fold(wt)
    if wf is None:
        raise RuntimeError("upconv_fold rejected the workload's weight")
    set_bytes = 2 * (x0.numel() + w.out_pixels * w.Cout)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = buffer_sets_for(set_bytes, l2, cap=8)
    sets = [(x0.clone(), torch.empty((w.N, 2 * w.H, 2 * w.W, w.Cout), dtype=torch.bfloat16, device=device))
            for _ in range(nsets)]
    h = stream.cuda_stream
    bptr = b.data_ptr() if b is not None else 0

    def call(i):
        x, y = sets[i]
        rc = gs.raw_gn_upconv_nhwc(x.data_ptr(), wf.data_ptr(), bptr, y.data_ptr(), w.N, w.H, w.W, w.Cin, w.Cout,
                                   stream=h)
        if rc != 0:
            raise RuntimeError(gs.status_string(rc))

    with torch.cuda.stream(stream):
        for i in range(5):
            call(i % nsets)
        torch.cuda.synchronize()
        per, _ = time_calls(call, nsets, max(10, steps // 2), stream)
        graph = capture_steps(call, nsets, steps, stream)
        graph.replay()
        elapsed = time_graph(graph, stream)
        del graph
    if gs.gn_device_status(False) != 0:
        raise RuntimeError("a bounded wait expired inside the upconv kernel")
    us = elapsed * 1e6 / steps
    tflops = w.flops / (us * 1e-6) / 1e12
    launch_us = statistics.mean(per) * 1e3
    out = {"workload": w.name, "us_per_call": round(us, 2), "tflops": round(tflops, 1),
           "frac": round(tflops / peak, 3), "launch_us_mean": round(launch_us, 2),
           "tflops_per_launch": round(w.flops / (launch_us * 1e-6) / 1e12, 1),
           "l2": f"{nsets} rotating (x, y) sets of {set_bytes >> 20} MiB", "launch": "cuda-graph"}
    if cudnn_context:
        # context only: PyTorch's own (cuDNN) upsample + conv2d on the same channels_last tensors
        xc = x0.permute(0, 3, 1, 2)

        def unfused(_):
            F.conv2d(F.interpolate(xc, scale_factor=2, mode="nearest"), wt, b, padding=1)
        with torch.cuda.stream(stream):
            unfused(0)
            torch.cuda.synchronize()
            pt, _ = time_calls(unfused, 1, 10, stream)
        out["torch_interpolate_conv2d_us"] = round(statistics.median(pt) * 1e3, 1)
        # the page's own formulation: ConvTranspose2d(k4, s2, p1) with the summed 4x4 taps
        # (kernel row k of the transposed conv sums 3x3 rows (2,), (1, 2), (0, 1), (0,))
        rows = ((2,), (1, 2), (0, 1), (0,))
        wt32 = wt.float()
        w4 = torch.zeros((w.Cin, w.Cout, 4, 4), dtype=torch.float32, device=device)
        for k1, r1 in enumerate(rows):
            for k2, r2 in enumerate(rows):
                for ky in r1:
                    for kx in r2:
                        w4[:, :, k1, k2] += wt32[:, :, ky, kx].t()
        w4 = w4.to(torch.bfloat16)

        def transposed(_):
            F.conv_transpose2d(xc, w4, b, stride=2, padding=1)
        with torch.cuda.stream(stream):
            transposed(0)
            torch.cuda.synchronize()
            pt, _ = time_calls(transposed, 1, 10, stream)
        out["torch_conv_transpose2d_us"] = round(statistics.median(pt) * 1e3, 1)
    del sets
    torch.cuda.empty_cache()
    return out


def upconv_cpu_baseline(w, budget_s=10.0):
    """The fp64 oracle on sampled outputs of the workload, in the metric's
    unit (folded multiply-adds per second), on the host's cores."""
    import numpy as np
    import oracle
    from channels_last_groupnorm_gb300 import workloads as wl
    c = wl.make_upconv_inputs(w)
    orc = oracle.upconv()
    total = w.out_pixels * w.Cout
    rng = np.random.default_rng(0)
    count = 256
    while True:
        idx = rng.integers(0, total, count)
        t0 = time.perf_counter()
        orc.at(c["x_bits"], c["w_bits"], c["bias_bits"], idx)
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or count >= 1 << 22:
            break
        count *= 4
    rate = count * 2 * 4 * w.Cin / dt / 1e12
    return {"value": round(rate, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{count} randomly chosen outputs of {w.name} (of {total}), each a direct fp64 sum over "
                      f"its 9 Cin upsampled-window terms, counted at the folded 4 Cin multiply-adds"}


def run_upconv(args, w, device, rank, world):
    """One upsample + conv workload on its own: the line reports its TFLOP/s
    against the measured bf16 tensor peak."""
    import torch
    from channels_last_groupnorm_gb300 import gnsilu as gs
    stream = torch.cuda.Stream(device)
    peak, peak_kind, sustained = tensor_peak()
    sampler = ClockSampler(device.index or 0) if rank == 0 else None
    if sampler:
        sampler.start()
    r = measure_upconv(w, args.steps, device, stream, peak, cudnn_context=not args.no_sweep)
    clocks = sampler.stop() if sampler else None
    elapsed_s = r["us_per_call"] * 1e-6 * args.steps
    total_elapsed, total_flops = reduce_timing(elapsed_s, float(w.flops) * args.steps,
                                               device=device if world > 1 else None)
    value = total_flops / total_elapsed / 1e12
    e2e = None
    if not args.no_e2e:
        e2e = measure_upconv_e2e(w, max(3, args.steps // 10), device, stream)
    line = {
        "metric": UPCONV_METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["us_per_call"] / 1e3, 6),
        "us_per_call": r["us_per_call"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "accumulate": "f32", "data": "synthetic (seeded numpy PCG64; x~N(0,1), "
        "w, bias ~U(-1/sqrt(9Cin), 1/sqrt(9Cin)), bf16)",
        "config": {**w.describe(), "l2": r["l2"], "launch": r["launch"],
                   "flops_per_step": "2 * N*2H*2W * Cout * 4 Cin (folded taps)"},
        "roofline": {"bound": "tensor", "achieved": r["tflops_per_launch"], "peak": peak, "unit": "TFLOP/s",
                     "frac": round(r["tflops_per_launch"] / peak, 4), "peak_kind": peak_kind,
                     "peak_sustained": sustained,
                     "traffic": recorded_traffic(w.name, "upconv", UPCONV_SOURCES),
                     "kernel": "upconv_kernel", "algorithmic_flops_per_launch": w.flops,
                     "launch_us_mean": r["launch_us_mean"]},
        "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks,
    }
    if "torch_interpolate_conv2d_us" in r:
        line["context"] = {"torch_interpolate_conv2d_us": r["torch_interpolate_conv2d_us"],
                           "torch_conv_transpose2d_us": r.get("torch_conv_transpose2d_us"),
                           "note": "PyTorch (cuDNN) on the same tensors and GPU: upsample + conv2d, and "
                                   "the summed-tap ConvTranspose2d(k4, s2, p1) the page runs"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = upconv_cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_upconv_e2e(w, steps, device, stream):
    """The same call end to end from pinned host buffers: x copied in, the
    kernel, y copied back, all inside the timed region (the folded weight
    stays resident, as a model's weights do)."""
    import torch
    from channels_last_groupnorm_gb300 import gnsilu as gs
    _, x0, wt, b = upconv_device_inputs(w, device)
    wf = gs.upconv_fold(wt)
    hx = x0.cpu().pin_memory()
    hy = torch.empty((w.N, 2 * w.H, 2 * w.W, w.Cout), dtype=torch.bfloat16).pin_memory()
    dx = torch.empty_like(x0)
    dy = torch.empty((w.N, 2 * w.H, 2 * w.W, w.Cout), dtype=torch.bfloat16, device=device)
    h = stream.cuda_stream
    bptr = b.data_ptr() if b is not None else 0

    def step(_):
        dx.copy_(hx, non_blocking=True)
        rc = gs.raw_gn_upconv_nhwc(dx.data_ptr(), wf.data_ptr(), bptr, dy.data_ptr(), w.N, w.H, w.W, w.Cin,
                                   w.Cout, stream=h)
        if rc != 0:
            raise RuntimeError(gs.status_string(rc))
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step(0)
        torch.cuda.synchronize()
        _, elapsed = time_calls(step, 1, steps, stream)
    us = elapsed * 1e6 / steps
    return {"value": round(w.flops / (us * 1e-6) / 1e12, 1), "unit": "TFLOP/s",
            "h2d_bytes_per_step": 2 * x0.numel(), "d2h_bytes_per_step": 2 * dy.numel(),
            "us_per_call": round(us, 1)}


def attn_device_inputs(w, device):
    import numpy as np
    import torch
    from channels_last_groupnorm_gb300 import workloads as wl
    c = wl.make_attn_inputs(w)

    def dev(bits):
        if bits is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)
    return c, {n: dev(c[n]) for n in c}


def measure_attn(w, steps, device, stream, peak, torch_context=True, schedule=None):
    """gn_attn_folded_ex on one mid-block attention workload: the weights
    are folded once (gn_attn_fold, untimed: per model), then a CUDA graph of
    `steps` calls is replayed.  ``schedule`` (default: the library's
    automatic choice) is reported with the kernels one call launches: the
    one-pass schedule keeps the scores on chip (2 launches, 3 when tiles are
    split between CTA pairs), the
    stored-weights one writes and reads the 2 S^2 bytes of softmax weights
    (5 launches; more than L2 at S = 16384).  TFLOP/s counts the folded
    evaluation: 2 S D^2 (value rows) + 4 S^2 D (scores, weighted sum)."""
    import torch
    import torch.nn.functional as F
    from channels_last_groupnorm_gb300 import gnsilu as gs
    if schedule is None:
        schedule = gs.ATTN_AUTO
    _, t = attn_device_inputs(w, device)
    wf, bf = gs.attn_fold(t["wv"], t["bv"], t["wo"], t["bo"])
    out = torch.empty_like(t["q"])
    need = gs.gn_attn_workspace_bytes(w.S, w.D)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    h = stream.cuda_stream
    rptr = t["residual"].data_ptr() if t["residual"] is not None else 0

    def call(_):
        rc = gs.raw_gn_attn_folded_ex(t["q"].data_ptr(), t["k"].data_ptr(), t["xn"].data_ptr(), wf.data_ptr(),
                                      bf.data_ptr(), rptr, out.data_ptr(), w.S, w.D, ws.data_ptr(), need,
                                      schedule, stream=h)
        if rc != 0:
            raise RuntimeError(gs.status_string(rc))

    torch.cuda.synchronize()
    before = gs.gn_kernel_launch_count()
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    kernels = int(gs.gn_kernel_launch_count() - before)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call(0)
        torch.cuda.synchronize()
        per, _ = time_calls(call, 1, max(5, steps // 2), stream)
        graph = capture_steps(call, 1, steps, stream)
        graph.replay()
        elapsed = time_graph(graph, stream)
        del graph
    if gs.gn_device_status(False) != 0:
        raise RuntimeError("a bounded wait expired inside the attention kernels")
    us = elapsed * 1e6 / steps
    launch_us = statistics.mean(per) * 1e3
    r = {"workload": w.name, "us_per_call": round(us, 2), "tflops": round(w.flops / (us * 1e-6) / 1e12, 1),
         "frac": round(w.flops / (us * 1e-6) / 1e12 / peak, 3), "launch_us_mean": round(launch_us, 2),
         "tflops_per_call_events": round(w.flops / (launch_us * 1e-6) / 1e12, 1),
         "kernels_per_call": kernels, "schedule": "stored_weights" if kernels == 5 else "one_pass",
         "workspace_bytes": need, "launch": "cuda-graph"}
    if torch_context:
        # context only: the stock block (value projection, SDPA, output projection, residual) in PyTorch
        def stock(_):
            v = F.linear(t["xn"], t["wv"], t["bv"])
            o = F.scaled_dot_product_attention(t["q"][None, None], t["k"][None, None], v[None, None])[0, 0]
            y = F.linear(o, t["wo"], t["bo"])
            if t["residual"] is not None:
                y = y + t["residual"]
            return y
        with torch.cuda.stream(stream):
            stock(0)
            torch.cuda.synchronize()
            pt, _ = time_calls(stock, 1, 5, stream)
        r["torch_linear_sdpa_linear_us"] = round(statistics.median(pt) * 1e3, 1)
    del ws
    torch.cuda.empty_cache()
    return r


def attn_cpu_baseline(w, budget_s=10.0):
    """The fp64 oracle on sampled query rows, in the metric's unit (folded
    multiply-adds per second): the value projection of all S rows, then the
    sampled rows' attention."""
    import numpy as np
    import oracle
    from channels_last_groupnorm_gb300 import workloads as wl
    c = wl.make_attn_inputs(w)
    orc = oracle.attn()
    args = (c["q"], c["k"], c["xn"], c["wv"], c["bv"], c["wo"], c["bo"], c["residual"])
    rows = 4
    while True:
        idx = np.random.default_rng(0).integers(0, w.S, rows)
        t0 = time.perf_counter()
        orc.rows(*args, idx)
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or rows >= w.S:
            break
        rows = min(w.S, rows * 4)
    flops = 2 * w.S * w.D * w.D + rows * 4 * w.S * w.D
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows} query rows of {w.name} (of {w.S}) after the value projection of all rows, fp64, "
                      f"unfolded; counted at the folded multiply-adds of that work"}


def run_attn(args, w, device, rank, world):
    import torch
    stream = torch.cuda.Stream(device)
    peak, peak_kind, sustained = tensor_peak()
    sampler = ClockSampler(device.index or 0) if rank == 0 else None
    if sampler:
        sampler.start()
    r = measure_attn(w, args.steps, device, stream, peak, torch_context=not args.no_sweep)
    clocks = sampler.stop() if sampler else None
    elapsed_s = r["us_per_call"] * 1e-6 * args.steps
    total_elapsed, total_flops = reduce_timing(elapsed_s, float(w.flops) * args.steps,
                                               device=device if world > 1 else None)
    line = {
        "metric": ATTN_METRIC, "value": round(total_flops / total_elapsed / 1e12, 1), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["us_per_call"] / 1e3, 6), "us_per_call": r["us_per_call"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "f32", "data": "synthetic (seeded numpy PCG64; q, k, xn, residual ~N(0,1); "
        "W, b ~U(-1/sqrt(D), 1/sqrt(D)); bf16)",
        "config": {**w.describe(), "launch": r["launch"], "workspace_bytes": r["workspace_bytes"],
                   "schedule": r["schedule"],
                   "flops_per_step": "2 S D^2 + 4 S^2 D (folded value rows, scores, weighted sum)"},
        "roofline": {"bound": "tensor", "achieved": r["tflops_per_call_events"], "peak": peak,
                     "unit": "TFLOP/s", "frac": round(r["tflops_per_call_events"] / peak, 4),
                     "peak_kind": peak_kind, "peak_sustained": sustained,
                     "traffic": recorded_traffic(w.name, "attn_" + r["schedule"], ATTN_SOURCES),
                     "kernel": ("whole call: the value-row gemm_kernel + attn_flash_kernel" if r["schedule"] == "one_pass"
                                else "whole call: 4 gemm_kernel launches + softmax_stats_kernel")
                               + " (shares in the committed ncu launch list); traffic = DRAM bytes of the "
                               + f"{r['kernels_per_call']} per call",
                     "algorithmic_flops_per_launch": w.flops, "launch_us_mean": r["launch_us_mean"]},
        "e2e": None, "gpu_launches": r["kernels_per_call"] * args.steps, "clocks": clocks,
    }
    if "torch_linear_sdpa_linear_us" in r:
        line["context"] = {"torch_linear_sdpa_linear_us": r["torch_linear_sdpa_linear_us"],
                           "note": "PyTorch's stock block (value Linear, SDPA, output Linear, residual) on the "
                                   "same tensors and GPU"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = attn_cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    from channels_last_groupnorm_gb300 import build as gnbuild
    from channels_last_groupnorm_gb300 import gnsilu as gs
    from channels_last_groupnorm_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(gnbuild.LIB_PATH):
        gnbuild.build()
    barrier()
    gs.lib()
    if args.workload in wl.RGA_BY_NAME:
        run_rga(args, wl.RGA_BY_NAME[args.workload], device, rank, world)
        return
    if args.workload in wl.UPCONV_BY_NAME:
        run_upconv(args, wl.UPCONV_BY_NAME[args.workload], device, rank, world)
        return
    if args.workload in wl.ATTN_BY_NAME:
        run_attn(args, wl.ATTN_BY_NAME[args.workload], device, rank, world)
        return
    w = wl.BY_NAME[args.workload]
    variant_id = {"auto": 0, "two_pass": 1, "fused": 2, "cluster": 3}[args.variant]
    stream = torch.cuda.Stream(device)
    peak, peak_kind = hbm_peak()

    sampler = ClockSampler(local) if rank == 0 else None
    r = measure_workload(w, variant_id, args.steps, args.warmup, device, stream,
                         soak_s=args.soak, sampler=sampler, launch=args.launch)
    ms_per_step = r["elapsed_s"] * 1e3 / args.steps
    units = 4.0 * w.elements * args.steps
    elapsed, total_units = reduce_timing(r["elapsed_s"], units,
                                         device=device if world > 1 else None)
    value = total_units / elapsed / 1e9

    per = r["per_step_ms"]
    launch_ms = statistics.mean(per)
    alg_bytes = 4.0 * w.elements
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    traffic = recorded_traffic(w.name, r["variant"])

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(5, args.steps // 2)
        e2e_s, h2d, d2h = measure_e2e(w, variant_id, e2e_steps, args.warmup, device, stream)
        e2e_elapsed, e2e_units = reduce_timing(e2e_s, 4.0 * w.elements * e2e_steps,
                                               device=device if world > 1 else None)
        e2e = {"value": round(e2e_units / e2e_elapsed / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "us_per_call": round(e2e_s * 1e6 / e2e_steps, 2)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_call": round(ms_per_step * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": (f"synthetic (seeded numpy PCG64; x~N({w.x_mean},{w.x_std}) bf16, gamma~U(0.5,1.5), "
                 "beta~N(0,0.1))"),
        "config": line_config(w, True, world),
        "schedule": {"variant": r["variant"], "launch": r["launch"],
                     "buffer_sets": f"{r['nsets']} rotating buffer sets of {r['set_bytes'] >> 20} MiB (x+y)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic,
                     "kernel": {"fused": "gn_fused_kernel", "cluster": "gn_cluster_kernel"}.get(
                         r["variant"], "pass1+finalize+pass2"),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "achieved_6B": round(1.5 * achieved, 1), "frac_6B": round(1.5 * achieved / peak, 4),
                     "launch_us_mean": round(launch_ms * 1e3, 3),
                     "launch_us_median": round(statistics.median(per) * 1e3, 3)},
        "e2e": e2e,
        "gpu_launches": int(r["launches"]),
        "clocks": r["clocks"],
    }
    if w.pages_us_h200:
        pages_gbs = 4.0 * w.elements / (w.pages_us_h200 * 1e-6) / 1e9
        line["vs_baseline"] = round(value / (pages_gbs * world), 3)
        line["baseline_note"] = (f"pages' two-pass Triton kernel on H200: {w.pages_us_h200} us/call"
                                 f" = {pages_gbs:.1f} GB/s at 4 B/elem (context, other hardware)")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0 and not args.no_sweep:
        tpeak = tensor_peak()[0]
        line["residual_gate"] = [measure_rga(rw, fmt, 50, device, stream, peak)
                                 for rw in wl.RGA_WORKLOADS for fmt in ("bf16", "fp16")]
        line["upsample_conv"] = [measure_upconv(uw, 20, device, stream, tpeak)
                                 for uw in wl.UPCONV_WORKLOADS[1:]]
        line["attention_folded"] = [measure_attn(aw, 10, device, stream, tpeak)
                                    for aw in wl.ATTN_WORKLOADS[1:]]
        rows = sweep(variant_id, device, stream, peak, launch=args.launch)
        line["sweep"] = rows
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baselines"] = cpu_baselines()
        line["gn_sweep"] = compact_sweep(rows)
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_rga(args, w, device, rank, world):
    """One residual-gate workload (bf16) on its own: the line reports its
    bandwidth at 6 B/element; used for its profiles."""
    import torch
    stream = torch.cuda.Stream(device)
    peak, peak_kind = hbm_peak()
    r = measure_rga(w, "bf16", args.steps, device, stream, peak)
    if rank == 0:
        print(json.dumps({
            "metric": "residual + gate*update bf16 us/call and HBM GB/s (6 B/elem)", "value": r["gbs_6B"],
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "us_per_call": r["us_per_call"], "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": w.describe(),
            "roofline": {"bound": "hbm", "achieved": r["gbs_6B"], "peak": peak, "unit": "GB/s",
                         "frac": r["frac_6B"], "peak_kind": peak_kind, "traffic": None,
                         "kernel": "rga_kernel", "algorithmic_bytes_per_launch": 6.0 * w.elements},
        }), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from channels_last_groupnorm_gb300 import workloads as wl
    if args.workload in wl.ATTN_BY_NAME:
        aw = wl.ATTN_BY_NAME[args.workload]
        attn_cpu_baseline(aw, budget_s=2.0)
        cb = attn_cpu_baseline(aw, budget_s=min(40.0, 100.0 / max(1, args.steps)))
        print(json.dumps({
            "impl": "reference", "metric": ATTN_METRIC, "value": cb["value"], "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": aw.describe(),
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    if args.workload in wl.UPCONV_BY_NAME:
        uw = wl.UPCONV_BY_NAME[args.workload]
        # warm-up: one untimed sample; then the timed sample sized to ~10 s per step budget
        upconv_cpu_baseline(uw, budget_s=2.0)
        cb = upconv_cpu_baseline(uw, budget_s=min(40.0, 100.0 / max(1, args.steps)))
        print(json.dumps({
            "impl": "reference", "metric": UPCONV_METRIC, "value": cb["value"], "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": uw.describe(),
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    w = wl.BY_NAME[args.workload]
    case = wl.make_inputs(w)
    orc = oracle.get()
    cores = orc.max_threads()
    # size each step so that warm-up + steps take about two minutes at most
    t0 = time.perf_counter()
    orc.forward(case["x_bits"][:, : max(1, w.L // 16)], case["gamma"], case["beta"], w.G,
                w.eps, True)
    per_row = (time.perf_counter() - t0) / max(1, w.L // 16)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.L, budget / max(per_row, 1e-9))))
    sample = case["x_bits"][:, :rows]
    for _ in range(args.warmup):
        orc.forward(sample, case["gamma"], case["beta"], w.G, w.eps, True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.forward(sample, case["gamma"], case["beta"], w.G, w.eps, True)
    dt = (time.perf_counter() - t0) / args.steps
    value = 4.0 * w.N * rows * w.C / dt / 1e9
    desc = (f"fp64 oracle on the first {rows} of {w.L} rows of the {w.name} tensor "
            f"per step, {cores} OpenMP threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": line_config(w, True, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--variant", choices=["auto", "fused", "two_pass", "cluster"], default="auto")
    ap.add_argument("--launch", choices=["graph", "stream"], default="graph",
                    help="submit the timed steps as one captured CUDA graph, or one stream "
                         "launch per step")
    ap.add_argument("--soak", type=float, default=1.5,
                    help="seconds of untimed calls while the clock sampler runs")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end measurement (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
