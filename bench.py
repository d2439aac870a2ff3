#!/usr/bin/env python3
"""Throughput benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one fused attention forward (attn_fwd, one kernel launch) over the
B=1 h=16 S=4096 d=64 fp16 workload (contiguous [B,h,S,d], non-causal, scale
1/8).  Inputs are synthetic (seeded N(0,1)) and already resident in HBM when
the timed region starts; 8 input sets (256 MiB in total, above the 129 MB L2)
are rotated so that no step reads inputs another step left in L2.  Timing:
W untimed warm-up steps, then exactly K steps between CUDA events recorded on
the launching stream, with a barrier and a synchronize on both sides; the
maximum over ranks is taken.  value = total FLOPs of all ranks (4·B·h·S²·d per
step and rank) / that time.

Multi-GPU (torchrun, one rank per GPU): each rank runs its own independent
problem of the same size (the (batch, head) units of attention need no
exchange), so per-GPU work is fixed and scaling is weak.

Also reported, on rank 0:
  roofline      achieved TFLOP/s of the attention kernel vs the measured dense
                FP16/BF16 tensor peak, and DRAM traffic per launch from the
                committed ncu summary (null once the kernel source changed);
  e2e           the same metric through the C-ABI call with pinned HOST
                buffers: every step copies Q, K, V host->device and O back;
  cpu_baseline  the fp64 oracle timed on the host cores on a bounded sample
                of query rows of the same workload;
  extra         the unfused two-pass comparison path on the same workload and
                the other workloads' fused throughput.
``--impl reference`` times the oracle alone (CPU), on the same metric.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (4·B·h·S²·d) & % of GB300 FP16 tensor peak, 1 GPU"
UNIT = "TFLOP/s"
WORKLOAD = "mha_f16_s4096"
N_SETS = 8
STEADY_S = 1.2  # seconds of the steady-state run added when the timed region is shorter
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-extra", action="store_true", help="skip the comparison / other-workload lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--only", choices=["qkv", "qkv1", "naive", "mixed", "fused"],
                    help="run only this path's calls (for profiling): the BERT-base projection + attention "
                         "(qkv: two launches, qkv1: the single kernel), "
                         "the unfused two-pass path or the fp32-input path on the bench workload, or the fused "
                         "attention (attn_fwd with its balancing scratch) on --workload; prints its time per "
                         "call, not the benchmark line")
    ap.add_argument("--shape", help="with --only fused: B,h,S overriding the workload's sizes (e.g. 1,2,16384)")
    return ap.parse_args()


# ----------------------------------------------------------------- ranks ----
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Maximum of a host float over all ranks (one all-reduce; host-side
    timing only -- the attention itself has no collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(w, rank: int, set_index: int) -> int:
    """Seed of input set `set_index` on `rank`: every rank draws its own problem."""
    return w.seed * 100 + set_index + 1000 * rank


def aggregate_tflops(flops_per_step: float, steps: int, world: int, t_max: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of its own problem
    (weak scaling), timed by the slowest rank."""
    return flops_per_step * steps * world / t_max / 1e12


# ---------------------------------------------------------------- clocks ----
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling every 100 ms while the timed region runs."""

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].strip()[:1].isdigit()), default=None)}


def clocks_once(gpu_index):
    """One read-only nvidia-smi reading of the SM clock and throttle reasons."""
    try:
        r = subprocess.run(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                            "-i", str(gpu_index)], capture_output=True, text=True, timeout=10)
    except (OSError, subprocess.TimeoutExpired):
        return None
    row = [c.strip() for c in r.stdout.strip().split(",")]
    if len(row) < 9:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    try:
        return {"sm_mhz": float(row[1]), "sm_max_mhz": float(row[2]),
                "reasons": [names[i] for i in range(4) if "Active" in row[5 + i] and "Not" not in row[5 + i]]}
    except ValueError:
        return None


# ----------------------------------------------------------------- peaks ----
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=FALLBACK_PEAKS["bf16_tflops"], source="fallback")


def profile_traffic(kernel_hash):
    """DRAM bytes per launch of the attention kernel, copied from the ncu
    capture recorded in profiles/flash_fwd_<workload>.json, if that capture was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"flash_fwd_{WORKLOAD}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_hash:
        return None
    try:
        return int(rec["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


# -------------------------------------------------------------- CPU legs ----
def oracle_rows_timing(w, q, k, v, n_rows, nthreads=0, seed=3):
    """Times the oracle on n_rows sampled query rows; returns (seconds, flops, threads)."""
    import oracle
    from head_attention_fwd_gb300.inputs import sample_rows

    rows = sample_rows(w, n_rows, seed=seed).numpy()
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows, layout=w.layout, scale=w.scale, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, 4.0 * w.S * w.d * len(rows), oracle.threads(nthreads)


def cpu_baseline(w, q, k, v, budget_s=12.0):
    """The oracle as it stands, on all host cores, on about budget_s of work."""
    import oracle
    cores = oracle.threads(0)
    dt, fl, _ = oracle_rows_timing(w, q, k, v, max(cores, 32))
    per_row = dt / max(cores, 32)
    n = int(min(w.B * w.h * w.S, max(cores, budget_s / max(per_row, 1e-6))))
    dt, fl, thr = oracle_rows_timing(w, q, k, v, n)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"{n} of {w.B * w.h * w.S} query rows of {w.name} (seeded sample), fp64, "
                      f"{dt:.1f} s"}


# ------------------------------------------------------------- our path ----
def time_graph(fn, n_inner, n_rep):
    """Seconds per call of fn(i) replayed from a CUDA graph that holds n_inner
    calls (the calls' host-side argument handling is paid once, at capture).
    fn must launch on torch's current stream."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(2):
            fn(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n_inner):
            fn(i)
    graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(n_rep):
        graph.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3 / (n_inner * n_rep)


def time_launches(fn, n, stream):
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(n):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def run_ours(args):
    import torch

    import head_attention_fwd_gb300 as attn
    from head_attention_fwd_gb300 import _build
    from head_attention_fwd_gb300.inputs import WORKLOADS, make_qkv

    world, rank, local = dist_init(args.gpus)
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    stream = torch.cuda.current_stream()

    # N_SETS independent input sets, generated on the device from fixed seeds.
    g = torch.Generator(device=dev)
    sets = []
    for i in range(N_SETS):
        g.manual_seed(rank_seed(w, rank, i))
        q, k, v = (torch.randn(w.shape(), generator=g, device=dev, dtype=torch.float32).to(w.torch_dtype)
                   for _ in range(3))
        sets.append((q, k, v, torch.empty_like(q)))
    set_bytes = sum(t.numel() * t.element_size() for t in sets[0])
    ws = split_scratch(attn, w, dev)

    def step(i):
        q, k, v, o = sets[i % N_SETS]
        attn.attn_fwd(q, k, v, o, layout=w.layout, stream=stream, workspace=ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    rc, detail = attn.attn_get_device_status()
    if rc:
        raise RuntimeError(f"device status after warm-up: {attn.attn_status_string(rc)} ({detail:#x})")

    sampler = ClockSampler(local) if rank == 0 else None
    before = clocks_once(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    t_local = time_launches(step, args.steps, stream)
    barrier(world)
    torch.cuda.synchronize()
    after = clocks_once(local) if rank == 0 else None
    clocks = sampler.stop() if sampler else None
    t = max_over_ranks(t_local, world)
    rc, detail = attn.attn_get_device_status()
    if rc:
        raise RuntimeError(f"device status after timed region: {attn.attn_status_string(rc)}")

    # A timed region shorter than about a second holds too few clock samples
    # (the sampler reads every 100 ms): time the same call again over at least
    # a second, with its own clock samples, as steady-state evidence.
    steady = None
    if t_local < STEADY_S:
        n_st = int(math.ceil(STEADY_S / (t_local / args.steps)))
        st_sampler = ClockSampler(local) if rank == 0 else None
        t_st = time_launches(step, n_st, stream)
        st_clocks = st_sampler.stop() if st_sampler else None
        steady = {"value": aggregate_tflops(w.attn_flops, n_st, 1, t_st), "unit": UNIT, "steps": n_st,
                  "ms_per_step": t_st / n_st * 1e3, "seconds": t_st, "clocks": st_clocks}
    if rank == 0 and (clocks is None or not clocks.get("samples")):
        src = steady["clocks"] if steady and steady["clocks"] else {}
        reasons = sorted(set(src.get("reasons", [])) | set((before or {}).get("reasons", []))
                         | set((after or {}).get("reasons", [])))
        clocks = {"sm_mhz": src.get("sm_mhz", (after or before or {}).get("sm_mhz")),
                  "sm_max_mhz": src.get("sm_max_mhz", (after or before or {}).get("sm_max_mhz")),
                  "reasons": reasons, "samples": 0, "before": before, "after": after,
                  "note": (f"the {t_local * 1e3:.1f} ms timed region held no 100 ms sample; sm_mhz and reasons "
                           "come from the steady-state run of the same call and from one reading "
                           "right before and after the timed region")}
    elif clocks is not None:
        clocks["before"], clocks["after"] = before, after

    flops_step = w.attn_flops
    value = aggregate_tflops(flops_step, args.steps, world, t)
    kernel_tflops = flops_step * args.steps / t_local / 1e12

    if rank != 0:
        barrier(world)
        return

    peaks = measured_peaks()
    alg_bytes = 4 * w.B * w.h * w.S * w.d * torch.tensor([], dtype=w.torch_dtype).element_size()
    khash = _build.source_hash()
    roofline = {
        "bound": "tensor", "achieved": kernel_tflops, "peak": peaks["bf16_tflops"], "unit": UNIT,
        "frac": kernel_tflops / peaks["bf16_tflops"], "traffic": profile_traffic(khash),
        "peak_source": f"{peaks['source']} dense bf16 burst (fp16 runs at the bf16 rate)",
        "frac_of_sustained": kernel_tflops / peaks["bf16_tflops_sustained"],
        "hbm_gbs_algorithmic": alg_bytes / (t_local / args.steps) / 1e9,
        "hbm_frac": alg_bytes / (t_local / args.steps) / 1e9 / peaks["hbm_gbs"],
        "alg_bytes_per_launch": alg_bytes, "flops_per_launch": flops_step,
        "kernel_source_hash": khash,
    }

    e2e = run_e2e(attn, w, sets, stream, flops_step, args.steps, ws)

    extra = {}
    if not args.no_extra and world == 1:
        extra = run_extra(attn, w, sets, stream, dev)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "h": w.h, "S": w.S, "d": w.d, "layout": "BHSD",
                   "causal": False, "scale": w.scale, "global_batch": w.B * world,
                   "parallelism": f"independent problem per rank x{world} (no collective)",
                   "l2": f"{N_SETS} rotating input sets, {N_SETS * set_bytes / 2**20:.0f} MiB > 129 MB L2",
                   "schedule": ("persistent; last waves cut along keys "
                                f"({ws.numel() / 2**20:.1f} MiB scratch, attn_fwd_ws)") if ws is not None
                   else "persistent; whole items (attn_fwd)"},
        "gpu_launches": args.steps,
        "roofline": roofline,
        "clocks": clocks,
        "e2e": e2e,
        "pct_of_tensor_peak": 100.0 * kernel_tflops / peaks["bf16_tflops"],
    }
    if world == 1 and not args.no_cpu:
        from head_attention_fwd_gb300.inputs import make_qkv as mk
        qc, kc, vc = mk(w)
        line["cpu_baseline"] = cpu_baseline(w, qc, kc, vc)
    if steady:
        extra["steady_state"] = steady
    if extra:
        line["extra"] = extra
    print(json.dumps(line), flush=True)
    barrier(world)


def run_e2e(attn, w, sets, stream, flops_step, steps, ws):
    """The same metric through the public call with pinned HOST buffers: every
    step uploads its Q, K, V (H2D) and downloads its O (D2H) inside the timed
    region.  As a user of the library would, the steps are pipelined over two
    device buffer sets and three streams (upload, compute, download), so the
    copies of neighbouring steps overlap the current kernel."""
    import torch

    nb = 2
    # Q, K, V of a step side by side in one pinned buffer and one device
    # buffer, so that a step is one 24 MiB upload rather than three
    host_in = [torch.stack([t.cpu() for t in sets[i][:3]]).pin_memory() for i in range(nb)]
    host_out = [torch.empty_like(sets[0][0], device="cpu").pin_memory() for _ in range(nb)]
    dev_in = [torch.empty_like(host_in[0], device=sets[0][0].device) for _ in range(nb)]
    dev_sets = [(dev_in[b][0], dev_in[b][1], dev_in[b][2], torch.empty_like(sets[0][0])) for b in range(nb)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(nb)]
    ev_comp = [torch.cuda.Event() for _ in range(nb)]
    ev_down = [torch.cuda.Event() for _ in range(nb)]

    def step(i):
        b = i % nb
        qd, kd, vd, od = dev_sets[b]
        with torch.cuda.stream(up):
            up.wait_event(ev_comp[b])            # the kernel of step i-nb has read this set
            dev_in[b].copy_(host_in[b], non_blocking=True)
            ev_up[b].record(up)
        stream.wait_event(ev_up[b])
        stream.wait_event(ev_down[b])            # O of step i-nb has been downloaded
        attn.attn_fwd(qd, kd, vd, od, layout=w.layout, stream=stream, workspace=ws)
        ev_comp[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_comp[b])
            host_out[b].copy_(od, non_blocking=True)
            ev_down[b].record(down)

    for b in range(nb):  # events start out recorded (nothing pending)
        ev_comp[b].record(stream)
        ev_down[b].record(stream)
    n = max(20, min(steps, 500))
    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    up.wait_event(start)
    down.wait_event(start)
    for i in range(n):
        step(i)
    stream.wait_stream(up)
    stream.wait_stream(down)
    end.record(stream)
    torch.cuda.synchronize()
    t = start.elapsed_time(end) / 1e3
    return {"value": flops_step * n / t / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": host_in[0].numel() * host_in[0].element_size(),
            "d2h_bytes_per_step": host_out[0].numel() * host_out[0].element_size(),
            "pipeline": "upload / compute / download streams over 2 device buffer sets, one upload per step",
            "ms_per_step": t / n * 1e3}


def split_scratch(attn, w, dev):
    """Scratch that lets attn_fwd cut the last wave of items along the key
    axis (None when the item count already fills whole waves)."""
    import torch
    need = attn.attn_fwd_ws_bytes(w.B, w.h, w.S, w.d, w.torch_dtype)
    return torch.empty(need, dtype=torch.uint8, device=dev) if need else None


def run_extra(attn, w, sets, stream, dev):
    """Unfused comparison on the same workload and fused throughput on the
    other tensor-core workloads (each timed alone with CUDA events)."""
    import torch
    from head_attention_fwd_gb300.inputs import WORKLOADS

    out = {}
    q, k, v, o = sets[0]
    ws = torch.empty(attn.attn_fwd_naive_workspace_bytes(w.B, w.h, w.S, q.dtype), dtype=torch.uint8,
                     device=dev)
    for _ in range(3):
        attn.attn_fwd_naive(q, k, v, o, workspace=ws, layout=w.layout, stream=stream)
    n = 20
    t = time_launches(lambda i: attn.attn_fwd_naive(*sets[i % N_SETS], workspace=ws, layout=w.layout,
                                                    stream=stream), n, stream)
    out["naive_two_pass_" + w.name] = {"tflops": w.attn_flops * n / t / 1e12, "ms": t / n * 1e3,
                                       "launches_per_call": 4}
    del ws
    # the same workload through attn_fwd (whole items only, no scratch)
    for _ in range(3):
        attn.attn_fwd(q, k, v, o, layout=w.layout, stream=stream, split=False)
    n = 200
    t = time_launches(lambda i: attn.attn_fwd(*sets[i % N_SETS], layout=w.layout, stream=stream,
                                              split=False), n, stream)
    out[w.name + "_whole_items"] = {"tflops": w.attn_flops * n / t / 1e12, "ms": t / n * 1e3}
    # fp32 inputs, fp16 output: one conversion launch, then the fused kernel
    q32, k32, v32 = (x.float() for x in (q, k, v))
    wsm = torch.empty(attn.attn_fwd_mixed_workspace_bytes(w.B, w.h, w.S, w.d, q.dtype), dtype=torch.uint8,
                      device=dev)
    for _ in range(3):
        attn.attn_fwd_mixed(q32, k32, v32, o, workspace=wsm, out_dtype=q.dtype, layout=w.layout, stream=stream)
    n = 200
    t = time_launches(lambda i: attn.attn_fwd_mixed(q32, k32, v32, o, workspace=wsm, out_dtype=q.dtype,
                                                    layout=w.layout, stream=stream), n, stream)
    conv_bytes = 3 * q.numel() * (4 + 2)
    out["mixed_f32_in_" + w.name] = {"tflops": w.attn_flops * n / t / 1e12, "ms": t / n * 1e3,
                                     "launches_per_call": 2,
                                     "conversion_bytes": conv_bytes}
    del q32, k32, v32, wsm
    for name in ("long_seq_bf16_peaky", "wide_head_bf16_bshd"):
        ww = WORKLOADS[name]
        g = torch.Generator(device=dev).manual_seed(ww.seed)
        qq, kk, vv = (torch.randn(ww.shape(), generator=g, device=dev).to(ww.torch_dtype) for _ in range(3))
        oo = torch.empty_like(qq)
        lse = torch.empty((ww.B, ww.h, ww.S), dtype=torch.float32, device=dev) if ww.want_lse else None
        wsx = split_scratch(attn, ww, dev)
        for _ in range(3):
            attn.attn_fwd(qq, kk, vv, oo, lse, layout=ww.layout, stream=stream, workspace=wsx)
        n = 20
        t = time_launches(lambda i: attn.attn_fwd(qq, kk, vv, oo, lse, layout=ww.layout, stream=stream,
                                                  workspace=wsx), n, stream)
        out[name] = {"tflops": ww.attn_flops * n / t / 1e12, "ms": t / n * 1e3}
        del qq, kk, vv, oo, lse, wsx
    wb = WORKLOADS["bert_base_qkv"]
    g = torch.Generator(device=dev).manual_seed(wb.seed)
    x = torch.randn((wb.B, wb.S, wb.D), generator=g, device=dev).to(wb.torch_dtype)
    wq = (torch.randn((wb.D, 3 * wb.D), generator=g, device=dev) * wb.w_std).to(wb.torch_dtype)
    oo = torch.empty((wb.B, wb.S, wb.h, wb.d), dtype=wb.torch_dtype, device=dev)
    ws = torch.empty(attn.qkv_proj_attn_workspace_bytes(wb.B, wb.S, wb.D, x.dtype), dtype=torch.uint8,
                     device=dev)
    for _ in range(3):
        attn.qkv_proj_attn(x, wq, wb.h, oo, ws, stream=stream)
    n = 50
    t = time_launches(lambda i: attn.qkv_proj_attn(x, wq, wb.h, oo, ws, stream=stream), n, stream)
    fl = wb.attn_flops + wb.proj_flops
    # Back-to-back Python calls are host-bound at this size (about 30 us of GPU
    # work per call); replaying the calls from a CUDA graph gives the GPU rate.
    tg = time_graph(lambda i: attn.qkv_proj_attn(x, wq, wb.h, oo, ws, stream=torch.cuda.current_stream()),
                    20, 10)
    out["bert_base_qkv"] = {"tflops": fl / tg / 1e12, "ms": tg * 1e3,
                            "timing": "CUDA graph of 20 calls, replayed 10 times",
                            "tflops_eager": fl / (t / n) / 1e12, "ms_eager": t / n * 1e3,
                            "flops": "projection 2*B*S*D*3D + attention 4*B*h*S^2*d",
                            "launches_per_call": 2}
    # the same call as one kernel: projection tiles feed the attention on chip
    for _ in range(3):
        attn.qkv_proj_attn_fused(x, wq, wb.h, oo, stream=stream)
    t = time_launches(lambda i: attn.qkv_proj_attn_fused(x, wq, wb.h, oo, stream=stream), n, stream)
    tg = time_graph(lambda i: attn.qkv_proj_attn_fused(x, wq, wb.h, oo, stream=torch.cuda.current_stream()),
                    20, 10)
    out["bert_base_qkv_single_kernel"] = {"tflops": fl / tg / 1e12, "ms": tg * 1e3,
                                          "timing": "CUDA graph of 20 calls, replayed 10 times",
                                          "tflops_eager": fl / (t / n) / 1e12, "ms_eager": t / n * 1e3,
                                          "launches_per_call": 1}
    wc = WORKLOADS["single_head_f32"]
    g = torch.Generator(device=dev).manual_seed(wc.seed)
    qq, kk, vv = (torch.randn(wc.shape(), generator=g, device=dev) for _ in range(3))
    oo = torch.empty_like(qq)
    n = 200
    t = time_launches(lambda i: attn.attn_fwd(qq, kk, vv, oo, stream=stream), n, stream)
    tg = time_graph(lambda i: attn.attn_fwd(qq, kk, vv, oo, stream=torch.cuda.current_stream()), 20, 10)
    out["single_head_f32"] = {"us": t / n * 1e6, "us_graph": tg * 1e6,
                              "note": "latency-bound fp32 CUDA-core path; us: back-to-back Python calls, "
                                      "us_graph: replayed from a CUDA graph"}
    rc, detail = attn.attn_get_device_status()
    if rc:
        raise RuntimeError(f"device status after extra runs: {attn.attn_status_string(rc)}")
    return out


# ------------------------------------------------------- reference (CPU) ----
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from head_attention_fwd_gb300.inputs import WORKLOADS, make_qkv

    oracle.build()
    w = WORKLOADS[args.workload]
    q, k, v = make_qkv(w)
    cores = oracle.threads(0)
    # size each step so that the whole run stays within about two minutes
    dt, _, _ = oracle_rows_timing(w, q, k, v, max(cores, 32))
    per_row = dt / max(cores, 32)
    total_steps = args.steps + args.warmup
    rows = int(max(cores, min(w.B * w.h * w.S, 120.0 / max(per_row, 1e-7) / max(total_steps, 1))))
    for i in range(args.warmup):
        oracle_rows_timing(w, q, k, v, rows, seed=100 + i)
    t0 = time.perf_counter()
    fl = 0.0
    for i in range(args.steps):
        _, f, _ = oracle_rows_timing(w, q, k, v, rows, seed=1000 + i)
        fl += f
    t = time.perf_counter() - t0
    value = fl / t / 1e12
    sample = f"{rows} of {w.B * w.h * w.S} query rows of {w.name} per step (seeded), fp64"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / max(args.steps, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "h": w.h, "S": w.S, "d": w.d, "layout": "BHSD",
                   "causal": False, "scale": w.scale},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": cores, "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_only(args):
    """`--steps` calls of one secondary path after `--warmup` untimed ones, for
    ncu launch lists and captures of its kernels."""
    import torch

    import head_attention_fwd_gb300 as attn
    from head_attention_fwd_gb300 import _build
    from head_attention_fwd_gb300.inputs import WORKLOADS

    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    if args.only in ("qkv", "qkv1"):
        w = WORKLOADS["bert_base_qkv"]
        g = torch.Generator(device=dev).manual_seed(w.seed)
        x = torch.randn((w.B, w.S, w.D), generator=g, device=dev).to(w.torch_dtype)
        wq = (torch.randn((w.D, 3 * w.D), generator=g, device=dev) * w.w_std).to(w.torch_dtype)
        o = torch.empty((w.B, w.S, w.h, w.d), dtype=w.torch_dtype, device=dev)
        ws = torch.empty(attn.qkv_proj_attn_workspace_bytes(w.B, w.S, w.D, x.dtype), dtype=torch.uint8, device=dev)
        if args.only == "qkv":
            call = lambda i: attn.qkv_proj_attn(x, wq, w.h, o, ws, stream=stream)
        else:
            call = lambda i: attn.qkv_proj_attn_fused(x, wq, w.h, o, stream=stream)
        flops = w.attn_flops + w.proj_flops
    elif args.only == "fused":
        from head_attention_fwd_gb300.inputs import make_qkv
        w = WORKLOADS[args.workload]
        if args.shape:
            B, h, S = (int(x) for x in args.shape.split(","))
            w = w.with_(B=B, h=h, S=S)
        q, k, v = (t.to(dev) for t in make_qkv(w))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.h, w.S), dtype=torch.float32, device=dev) if w.want_lse else None
        ws = split_scratch(attn, w, dev) if w.dtype != "f32" else None
        call = lambda i: attn.attn_fwd(q, k, v, o, lse, layout=w.layout, stream=stream, workspace=ws)
        flops = w.attn_flops
    else:
        w = WORKLOADS[WORKLOAD]
        g = torch.Generator(device=dev).manual_seed(w.seed)
        q, k, v = (torch.randn(w.shape(), generator=g, device=dev).to(w.torch_dtype) for _ in range(3))
        o = torch.empty_like(q)
        flops = w.attn_flops
        if args.only == "naive":
            ws = torch.empty(attn.attn_fwd_naive_workspace_bytes(w.B, w.h, w.S, q.dtype), dtype=torch.uint8,
                             device=dev)
            call = lambda i: attn.attn_fwd_naive(q, k, v, o, workspace=ws, layout=w.layout, stream=stream)
        else:
            q, k, v = (x.float() for x in (q, k, v))
            ws = torch.empty(attn.attn_fwd_mixed_workspace_bytes(w.B, w.h, w.S, w.d, w.torch_dtype),
                             dtype=torch.uint8, device=dev)
            call = lambda i: attn.attn_fwd_mixed(q, k, v, o, workspace=ws, out_dtype=w.torch_dtype,
                                                 layout=w.layout, stream=stream)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    t = time_launches(call, args.steps, stream)
    rc, detail = attn.attn_get_device_status()
    if rc:
        raise RuntimeError(f"device status: {attn.attn_status_string(rc)} ({detail:#x})")
    print(json.dumps({"only": args.only, "workload": w.name, "B": w.B, "h": w.h, "S": w.S, "d": w.d,
                      "calls": args.steps, "ms_per_call": t / args.steps * 1e3,
                      "tflops": flops * args.steps / t / 1e12}), flush=True)


def main():
    args = parse_args()
    if args.only:
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
