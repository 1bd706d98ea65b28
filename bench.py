#!/usr/bin/env python
"""Benchmark: one MoE layer's forward + backward (dgrad and wgrad) on GB300.

A step is one pass of the whole hot path over one batch: route, dispatch
layout, permute, expert FFN forward, combine, combine backward, expert dgrad,
permute backward, router backward and expert wgrad, all through the C ABI on
one stream, with inputs already resident in HBM. The default workload is the
Qwen3-30B-A3B-shaped layer with forced-balanced routing (T=4096 tokens,
H=2048, 128 experts, top-8, SwiGLU inner 768), the configuration the pages
benchmark EP overlap on; data are synthetic (seeded, see moe_synth).

Prints one JSON line (rank 0). With --impl reference the CPU oracle is timed
instead, on a bounded token sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
Under torchrun (N > 1) each rank runs an independent replica (weak scaling,
no collective on the data path; the barrier and the max-over-ranks timing use
the process group).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 FMA lanes x 2 flop x 2.07 GHz (max SM clock)
FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# kernels whose floor is fp32 FMA arithmetic, not memory (fixed-order fp32 router sums)
ALU_BOUND = ("route_logits",)
# kernels whose floor is that arithmetic followed by their writes: the fused
# dispatch cannot write any x_perm row before the global expert counts exist,
# which needs every tile's routing, so its writes cannot overlap its FMA phase
ALU_THEN_WRITE = ("dispatch_fused",)


# ----------------------------------------------------------------------------- helpers
def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(d) -> dict:
    """Minimum bytes read, bytes written and flops per launch of each kernel.

    Bytes count each tensor the kernel must read or write once (the k-fold
    re-reads of x in the gathers are served by L2 and not counted); flops count
    multiply-adds as 2. Returns {kernel: (read_bytes, write_bytes, flops)}."""
    T, H, E, k, F = d["T"], d["H"], d["E"], d["k"], d["F"]
    N = T * k
    b2, b4 = 2, 4
    fused_topk = E <= 128  # the routing is fused into the logits kernel
    out = {
        "route_logits": (T * H * b2 + E * H * b2,
                         T * E * b4 + (2 * N * b4 if fused_topk else 0), 2.0 * T * H * E),
        "route_topk": (T * E * b4, 2 * N * b4, 0.0),
        # route + layout + permute in one launch: x and w_r read once; logits,
        # idx, gates, slot, row_src and x_perm written once
        "dispatch_fused": (T * H * b2 + E * H * b2,
                           T * E * b4 + 4 * N * b4 + N * H * b2 + (2 * E + 2) * b4,
                           2.0 * T * H * E),
        "layout_count": (N * b4, 0, 0.0),
        "layout_assign": (N * b4, 2 * N * b4, 0.0),
        "permute": (T * H * b2 + N * b4, N * H * b2, 0.0),
        "combine": (N * H * b2 + 2 * N * b4, T * H * b2, 2.0 * N * H),
        "combine_bwd": (T * H * b2 + N * H * b2 + 2 * N * b4, N * H * b2 + N * b4, 3.0 * N * H),
        "permute_bwd": (N * H * b2 + N * b4, T * H * b4, 1.0 * N * H),
        "route_bwd_dx": (T * H * b4 + E * H * b2 + 3 * N * b4, T * H * b2, 2.0 * N * H),
        # permute backward fused with the router's dx pass (the layer path)
        "dispatch_bwd": (N * H * b2 + 3 * N * b4 + E * H * b2, T * H * b2 + N * b4, 3.0 * N * H),
        # dW_r: chunk partials and their per-expert sum in one launch
        "route_bwd_dwr": (T * H * b2 + 2 * N * b4, E * H * b4, 2.0 * N * H),
        "gemm_fc1_fwd": (N * H * b2 + E * 2 * F * H * b2, N * 2 * F * b2 + N * F * b2,
                         2.0 * N * H * 2 * F),
        "gemm_fc2_fwd": (N * F * b2 + E * H * F * b2, N * H * b2, 2.0 * N * F * H),
        "gemm_fc2_dgrad": (N * H * b2 + E * H * F * b2 + N * 2 * F * b2, N * 2 * F * b2,
                           2.0 * N * H * F),
        "gemm_fc1_dgrad": (N * 2 * F * b2 + E * 2 * F * H * b2, N * H * b2, 2.0 * N * 2 * F * H),
        "gemm_wgrad_w1": (N * 2 * F * b2 + N * H * b2, E * 2 * F * H * b2, 2.0 * N * 2 * F * H),
        "gemm_wgrad_w2": (N * H * b2 + N * F * b2, E * H * F * b2, 2.0 * N * H * F),
    }
    # FC1 then FC2 forward, FC2 then FC1 dgrad, and the two weight gradients,
    # as one launch each
    for chain, (m1, m2) in (("gemm_ffn_fwd", ("gemm_fc1_fwd", "gemm_fc2_fwd")),
                            ("gemm_ffn_dgrad", ("gemm_fc2_dgrad", "gemm_fc1_dgrad")),
                            ("gemm_wgrad", ("gemm_wgrad_w1", "gemm_wgrad_w2"))):
        out[chain] = tuple(x + y for x, y in zip(out[m1], out[m2]))
    return out


def kernel_stats(agg: dict, algo: dict, pk: dict, wr_gbs: float) -> dict:
    """Per-kernel figures from {kernel: [launches, total ms]} and the
    algorithmic (read, write, flops) of each launch."""
    kernels = {}
    for name, (n, tot) in agg.items():
        avg_ms = tot / n
        rd, wr, fl = algo.get(name, (0.0, 0.0, 0.0))
        by = rd + wr
        # HBM floor: all bytes at the copy rate, or the written bytes at the
        # live write-only rate where that takes longer (a write-only stream is
        # faster than a copy on this part, so for these kernels it never does)
        t_floor = max(by / (pk["hbm_gbs"] * 1e9), wr / (wr_gbs * 1e9))
        gbs = by / (avg_ms * 1e-3) / 1e9 if avg_ms > 0 else 0.0
        tfl = fl / (avg_ms * 1e-3) / 1e12 if avg_ms > 0 else 0.0
        t_hbm = by / (pk["hbm_gbs"] * 1e9)
        t_tc = fl / (pk["bf16_tflops_sustained"] * 1e12) if name.startswith("gemm") else 0.0
        t_alu = fl / (FP32_TFLOPS * 1e12) if name in ALU_BOUND else 0.0
        bound = "tensor" if t_tc > t_hbm else "hbm"
        if t_alu > max(t_tc, t_hbm):
            bound = "alu"
        if name in ALU_THEN_WRITE:
            # FMA phase at the fp32 peak, then the writes at the write-only rate
            t_alu = fl / (FP32_TFLOPS * 1e12) + wr / (wr_gbs * 1e9)
            bound = "alu+write"
        t_bound = {"tensor": t_tc, "hbm": t_hbm, "alu": t_alu, "alu+write": t_alu}[bound]
        frac = t_bound / (avg_ms * 1e-3) if avg_ms > 0 else 0.0
        kernels[name] = {"launches": n, "avg_us": round(avg_ms * 1e3, 2),
                         "share": None, "GB_s": round(gbs, 1), "TFLOP_s": round(tfl, 1),
                         "bound": bound, "roofline_frac": round(frac, 3),
                         "hbm_floor_us": round(t_floor * 1e6, 1),
                         "hbm_floor_frac": round(t_floor / (avg_ms * 1e-3), 3) if avg_ms > 0 else None,
                         "algo_bytes": int(by), "algo_write_bytes": int(wr), "algo_flops": fl}
    return kernels


def accum_algorithmic(d) -> dict:
    """Bytes and flops of the weight-gradient GEMMs that add into fp32 main
    gradients: the operands, plus each main gradient read and written once."""
    T, H, E, k, F = d["T"], d["H"], d["E"], d["k"], d["F"]
    N = T * k
    w1, w2 = E * 2 * F * H * 4, E * H * F * 4
    return {"gemm_wgrad_w1_accum": (N * 2 * F * 2 + N * H * 2 + w1, w1, 2.0 * N * 2 * F * H),
            "gemm_wgrad_w2_accum": (N * H * 2 + N * F * 2 + w2, w2, 2.0 * N * H * F)}


def hbm_write_gbs(dev) -> float:
    """Write-only HBM bandwidth, measured live: best of 5 zero-fills of 1 GiB in
    8-byte elements (a fill of 1-byte elements issues narrow stores and reaches
    only about half the rate on this part)."""
    buf = torch.empty(1 << 27, dtype=torch.int64, device=dev)
    best = float("inf")
    for i in range(8):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        buf.zero_()
        e1.record()
        torch.cuda.synchronize(dev)
        if i >= 3:
            best = min(best, e0.elapsed_time(e1))
    del buf
    return (1 << 30) / (best * 1e-3) / 1e9


KERNEL_SOURCES = {  # the files each kernel family is built from
    "gemm": ("grouped_gemm.cu", "sm100_ptx.cuh", "moe_internal.cuh"),
    "route": ("route.cu", "moe_internal.cuh"),
    "layout": ("layout.cu", "moe_internal.cuh"),
    "permute": ("permute.cu", "moe_internal.cuh"),
    "combine": ("permute.cu", "moe_internal.cuh"),
    "dispatch": ("route.cu", "moe_internal.cuh"),
}


def code_only(text: str) -> str:
    """C/C++ source with comments and blank lines removed, trailing space trimmed
    (string literals are left as they are; none of the sources puts comment
    markers inside one)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def source_digest(kernel: str, read=None) -> str:
    """Hash of the code (comments stripped) of one kernel's sources: ncu traffic
    figures count only while it matches. read(name) -> text overrides the files."""
    files = KERNEL_SOURCES.get(kernel.split("_")[0], ())
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_router_softmax_top_gb300", "csrc")
    for f in files:
        if read is None:
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(f.encode() + code_only(text).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu record, or None if stale/absent."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        rec = t.get(workload, {}).get(kernel)
        if not rec or rec.get("source_digest") != source_digest(kernel):
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        try:
            bus = torch.cuda.get_device_properties(device).pci_bus_id
        except Exception:
            bus = str(device)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(bus), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def emit(obj):
    print(json.dumps(obj), flush=True)


# ----------------------------------------------------------------------------- oracle timing
_ORACLE_TIMER = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import moe_synth
from oracle import moe_oracle as O
inp = moe_synth.workload(sys.argv[2], T=int(sys.argv[3]))
t0 = time.perf_counter()
fwd = O.layer_forward(inp)
O.layer_backward(inp, fwd)
print(json.dumps({"seconds": time.perf_counter() - t0}))
"""


def oracle_timing(workload: str, T_sample: int, threads: int) -> dict:
    """Times the CPU oracle (fwd + bwd) on the first T_sample tokens of the
    workload in a fresh process limited to `threads` BLAS/OpenMP threads (the
    limit has to be set before numpy loads, hence the process)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[var] = str(threads)
    r = subprocess.run([sys.executable, "-c", _ORACLE_TIMER, ROOT, workload, str(T_sample)],
                       env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing failed: {r.stderr[-500:]}")
    sec = json.loads(r.stdout.strip().splitlines()[-1])["seconds"]
    return {"tokens_per_s": round(T_sample / sec, 3), "seconds": round(sec, 2), "threads": threads}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# ----------------------------------------------------------------------------- our arm
def _agg(prof):
    agg = {}
    for name, t in prof:
        a = agg.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += t
    return agg


def timed_steps(step, steps: int, st, groups: int = 10):
    """Times `steps` calls of step() between CUDA events on st; the events of
    `groups` equal slices give the step-to-step spread. Returns (ms per step,
    {min, median, max} ms per step over the slices)."""
    groups = max(1, min(groups, steps))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(groups + 1)]
    bounds = [round(i * steps / groups) for i in range(groups + 1)]
    ev[0].record(st)
    for g in range(groups):
        for _ in range(bounds[g + 1] - bounds[g]):
            step()
        ev[g + 1].record(st)
    torch.cuda.synchronize()
    total = ev[0].elapsed_time(ev[-1]) / steps
    per = [ev[g].elapsed_time(ev[g + 1]) / max(1, bounds[g + 1] - bounds[g])
           for g in range(groups)]
    return total, {"min": round(min(per), 4), "median": round(statistics.median(per), 4),
                   "max": round(max(per), 4), "groups": groups}


def profiled_kernels(moe, step, steps: int, per_step_launches: int, dev):
    """Per-launch durations of `steps` steps (events around each launch on its
    own stream), aggregated {kernel: [launches, total ms]}."""
    cap = per_step_launches * steps + 8
    moe.moe_profile_start(cap)
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    return _agg(moe.moe_profile_stop(cap))


def gemm_summary(kernels: dict, agg: dict, algo: dict, steps: int, pk: dict) -> dict:
    names = [n for n in kernels if n.startswith("gemm")]
    ms = sum(agg[n][1] for n in names) / steps
    fl = sum(algo[n][2] for n in names)
    tf = fl / (ms * 1e-3) / 1e12 if ms else None
    pc = [n for n in ("permute", "combine", "combine_bwd", "permute_bwd", "dispatch_bwd")
          if n in agg]
    pc_ms = sum(agg[n][1] for n in pc) / steps
    pc_bytes = sum(algo[n][0] + algo[n][1] for n in pc)
    return {"grouped_gemm_TFLOP_s": round(tf, 1) if tf else None,
            "grouped_gemm_frac_of_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 4)
            if tf else None,
            "permute_combine_GB_s": round(pc_bytes / (pc_ms * 1e-3) / 1e9, 1) if pc_ms else None}


def measure_workload(moe, wl: str, args, dev, st, pk, wr_gbs, steps: int) -> dict:
    """One single-micro-batch workload: the layer step timed, then every kernel
    timed in a profiled pass; the compact figures for the bench line."""
    import moe_synth
    inp = moe_synth.workload(wl)
    shape = inp.shape_dict()
    d = moe.LayerDesc.of(**shape)
    b = moe.LayerBuffers(d, dev)
    b.load_inputs(inp)
    torch.cuda.synchronize(dev)  # the loads ran on torch's stream, the steps run on st

    def step():
        moe.moe_layer_forward(d, b, st)
        moe.moe_layer_backward(d, b, True, st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    l0 = moe.moe_kernel_launches()
    step()
    torch.cuda.synchronize(dev)
    per_step = moe.moe_kernel_launches() - l0
    ms, spread = timed_steps(step, steps, st)
    agg = profiled_kernels(moe, step, min(steps, 20), per_step, dev)
    status = moe.moe_device_status(d, b.ws, st)
    if status != moe.MOE_OK:
        raise RuntimeError(f"{wl}: device status {status}: {moe.lib().moe_last_error()}")
    algo = algorithmic(shape)
    ks = kernel_stats(agg, algo, pk, wr_gbs)
    cnt = b.cnt.cpu()
    out = {"config": {"workload": wl, **shape}, "ms_per_step": round(ms, 4),
           "tokens_per_s": round(inp.T / (ms / 1e3), 1), "spread_ms_per_step": spread,
           "steps": steps, "rows_per_expert": {"min": int(cnt.min()), "max": int(cnt.max())},
           **gemm_summary(ks, agg, algo, min(steps, 20), pk),
           "kernels": {n: {k: v[k] for k in ("avg_us", "bound", "roofline_frac", "hbm_floor_frac",
                                             "GB_s", "TFLOP_s")} for n, v in ks.items()}}
    out["experts_by_rows"] = rows_histogram(cnt)
    del b
    torch.cuda.empty_cache()
    return out


BUCKET_ROWS = (64, 128, 256, 512, 1024, 2048, 4096)


def rows_histogram(cnt) -> dict:
    """Experts and their rows per bucket [M, 2M) of BUCKET_ROWS (the first
    bucket also takes fewer rows, the last more)."""
    hist = {}
    for i, m in enumerate(BUCKET_ROWS):
        lo = 0 if i == 0 else m
        hi = BUCKET_ROWS[i + 1] if i + 1 < len(BUCKET_ROWS) else 1 << 30
        sel = (cnt >= lo) & (cnt < hi)
        hist[str(m)] = {"experts": int(sel.sum()), "rows": int(cnt[sel].sum())}
    return hist


def measure_expert_buckets(moe, args, dev, st, pk, wr_gbs, skew_hist=None) -> dict:
    """Grouped-GEMM efficiency by rows per expert: all 128 experts of the
    Qwen3-30B-A3B-shaped layer (H=2048, F=768, k=8) with M rows each
    (T = 16 M tokens), for M in BUCKET_ROWS. The forward chain, the dgrad chain
    and the weight gradients are each timed through their C-ABI calls with
    CUDA events, on random operands, and rated against the same rooflines as
    in the layer step. The skewed workload's experts are counted into the same
    buckets, so its GEMM time can be read against these rates."""
    E, H, F, k = 128, 2048, 768, 8
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    rows = []
    for M in BUCKET_ROWS:
        T = E * M // k
        shape = {"T": T, "H": H, "E": E, "k": k, "F": F, "R": 1, "mode": 1}
        d = moe.LayerDesc.of(T=T, H=H, E=E, k=k, F=F)
        b = moe.LayerBuffers(d, dev)
        for t, std in ((b.x_perm, 1.0), (b.w1, 0.02), (b.w2, 0.02), (b.d_o, 0.01)):
            t.copy_(torch.randn(t.shape, generator=gen, device=dev, dtype=torch.float32) * std)
        b.off.copy_(torch.arange(E + 1, device=dev, dtype=torch.int32) * M)
        torch.cuda.synchronize(dev)  # the fills ran on torch's stream, the calls run on st
        calls = {
            "gemm_ffn_fwd": lambda: moe.moe_expert_ffn_fwd(d, b.x_perm, b.off, b.w1, b.w2, b.a, b.h,
                                                           b.o, b.ws, st),
            "gemm_ffn_dgrad": lambda: moe.moe_expert_ffn_bwd_dgrad(d, b.d_o, b.a, b.off, b.w1, b.w2,
                                                                   b.da, b.dx_perm, b.ws, st),
            "gemm_wgrad": lambda: moe.moe_expert_ffn_bwd_wgrad(d, b.x_perm, b.h, b.d_o, b.da, b.off,
                                                               b.dw1, b.dw2, b.ws, st),
        }
        n = max(3, 20 // max(1, M // 512))
        agg = {}
        for name, call in calls.items():  # in this order: each reads what the one before wrote
            for _ in range(max(args.warmup, 3)):
                call()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(n):
                call()
            e1.record(st)
            torch.cuda.synchronize(dev)
            agg[name] = [n, e0.elapsed_time(e1)]
        status = moe.moe_device_status(d, b.ws, st)
        if status != moe.MOE_OK:
            raise RuntimeError(f"buckets M={M}: device status {status}: "
                               f"{moe.lib().moe_last_error()}")
        algo = algorithmic(shape)
        ks = kernel_stats(agg, algo, pk, wr_gbs)
        ms = sum(v[1] / v[0] for v in agg.values())
        fl = sum(algo[nm][2] for nm in agg)
        row = {"rows_per_expert": M, "T": T,
               "TFLOP_s": round(fl / (ms * 1e-3) / 1e12, 1),
               "frac_of_bf16_sustained": round(fl / (ms * 1e-3) / 1e12
                                               / pk["bf16_tflops_sustained"], 3),
               "calls": {nm: {x: ks[nm][x] for x in ("avg_us", "bound", "roofline_frac",
                                                     "hbm_floor_frac", "TFLOP_s")}
                         for nm in agg}}
        if skew_hist is not None:
            row["skewed_layer"] = skew_hist[str(M)]
        rows.append(row)
        del b, calls
        torch.cuda.empty_cache()
    return {"note": "all 128 experts at M rows (T = 16 M); 'skewed_layer' counts the experts of "
                    "the skewed workload with rows in [M, 2M) (the first bucket also takes "
                    "fewer rows, the last more)",
            "buckets": rows}


def measure_schedule(moe, args, dev, steps: int) -> dict:
    """Two micro-batches of the balanced 4096-token layer: the serial schedule
    against the two-stream overlap, all without per-phase events (which would
    stop programmatic dependent launch between kernels), then one pass of each
    with the events on for the interval analysis: the union of the dispatch/
    combine phases, the union of the GEMM phases, and their intersection (the
    hidden communication), never a sum of durations."""
    import moe_synth
    wl = "two_microbatch"
    i0, i1 = moe_synth.workload(wl, 0), moe_synth.workload(wl, 1)
    d = moe.LayerDesc.of(**i0.shape_dict())
    b0 = moe.LayerBuffers(d, dev)
    b0.load_inputs(i0)
    b1 = moe.LayerBuffers(d, dev, weights=b0)
    b1.load_inputs(i1, weights=False)
    torch.cuda.synchronize(dev)  # the loads ran on torch's stream, the steps run on others
    sc = torch.cuda.Stream(device=dev, priority=-1)
    sg = torch.cuda.Stream(device=dev)
    res = {}

    def layer_pair():  # the plain layer calls, one micro-batch after the other
        for b in (b0, b1):
            moe.moe_layer_forward(d, b, sc)
            moe.moe_layer_backward(d, b, True, sc)

    for _ in range(args.warmup):
        layer_pair()
    ms, spread = timed_steps(layer_pair, steps, sc)
    res["layer_calls_x2"] = {"ms_per_step": round(ms, 4), "spread_ms_per_step": spread}
    # overlap = 2 overlaps only micro-batch 1's dispatch with micro-batch 0's
    # expert forward; "_split" gives that forward 96 of the SMs and the
    # dispatch the rest (the best split measured on this layer)
    for name, overlap, defer, gemm_sms in (("serial", 0, 0, 0), ("overlap", 1, 0, 0),
                                           ("overlap_defer", 1, 1, 0),
                                           ("overlap_dispatch", 2, 0, 0),
                                           ("overlap_dispatch_split", 2, 0, 96)):
        s = moe.Scheduler(d, sc, sg, gemm_sms=gemm_sms)
        s.set_phase_timing(False)
        for _ in range(args.warmup):
            s.step(b0, b1, overlap=overlap, defer_wgrad=bool(defer))
        ms, spread = timed_steps(lambda: s.step(b0, b1, overlap=overlap,
                                                defer_wgrad=bool(defer)), steps, sc)
        s.flush()
        # one more pass with the phase events on, for the interval analysis
        s.set_phase_timing(True)
        s.step(b0, b1, overlap=overlap, defer_wgrad=bool(defer))
        comm, gemm, hidden = moe.interval_overlap(s.timings())
        s.flush()
        torch.cuda.synchronize(dev)
        s.close()
        res[name] = {"ms_per_step": round(ms, 4), "spread_ms_per_step": spread,
                     "gemm_sms": gemm_sms,
                     "timed_pass": {"comm_union_ms": round(comm, 4),
                                    "gemm_union_ms": round(gemm, 4),
                                    "hidden_comm_ms": round(hidden, 4)}}
    for b in (b0, b1):
        if moe.moe_device_status(d, b.ws) != moe.MOE_OK:
            raise RuntimeError(f"schedule: device status: {moe.lib().moe_last_error()}")
    best = min(("overlap", "overlap_defer", "overlap_dispatch", "overlap_dispatch_split"),
               key=lambda n: res[n]["ms_per_step"])
    out = {"config": {"workload": wl, **i0.shape_dict(), "micro_batches": 2},
           "steps": steps, "schedules": res, "best_overlap": best,
           "tokens_per_s_best_overlap": round(2 * i0.T / (res[best]["ms_per_step"] / 1e3), 1),
           "overlap_vs_serial": round(res["serial"]["ms_per_step"] / res[best]["ms_per_step"], 4),
           "overlap_vs_layer_calls": round(res["layer_calls_x2"]["ms_per_step"]
                                           / res[best]["ms_per_step"], 4)}
    del b0, b1
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local):
    import moe_synth
    import combine_router_softmax_top_gb300 as moe
    from combine_router_softmax_top_gb300 import build

    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    inp = moe_synth.workload(args.workload, microbatch=rank)
    shape = inp.shape_dict()
    d = moe.LayerDesc.of(**shape)
    b = moe.LayerBuffers(d, dev)
    b.load_inputs(inp)
    torch.cuda.synchronize(dev)  # the loads ran on torch's stream, the steps run on st
    st = torch.cuda.Stream(device=dev)

    def step():
        moe.moe_layer_forward(d, b, st)
        moe.moe_layer_backward(d, b, True, st)

    for _ in range(args.warmup):
        step()
    status = moe.moe_device_status(d, b.ws, st)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status {status}: {moe.lib().moe_last_error()}")
    torch.cuda.synchronize(dev)
    l0 = moe.moe_kernel_launches()
    step()
    torch.cuda.synchronize(dev)
    per_step_launches = moe.moe_kernel_launches() - l0

    # ---- timed region (no per-launch events inside: they would sit between
    # the kernels and break programmatic dependent launch)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = moe.moe_kernel_launches()
    e0.record(st)
    for _ in range(args.steps):
        step()
    e1.record(st)
    torch.cuda.synchronize(dev)
    launches = moe.moe_kernel_launches() - launches0
    barrier(world)
    clk = clocks.stop()
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, world)

    # ---- the same step sustained for about a second, in event-timed slices,
    # with its own clock record: the spread and the clocks under a longer load
    sustained = None
    if not args.no_sustained:
        n_sus = max(args.steps, int(1.0 / max(ms_local * 1e-3, 1e-6)))
        clocks2 = ClockSampler(local)
        time.sleep(0.25)
        sms, spread = timed_steps(step, n_sus, st, groups=20)
        sustained = {"steps": n_sus, "ms_per_step": round(sms, 4), "spread_ms_per_step": spread,
                     "clocks": clocks2.stop()}

    # ---- per-kernel durations: the same steps again, each launch bracketed by
    # CUDA events on its own stream
    prof_steps = min(args.steps, 50)
    agg = profiled_kernels(moe, step, prof_steps, per_step_launches, dev)
    status = moe.moe_device_status(d, b.ws, st)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status {status}: {moe.lib().moe_last_error()}")
    tokens_per_s = world * inp.T / (ms / 1e3)

    # ---- per-kernel figures from the live events
    algo = algorithmic(shape)
    wr_gbs = hbm_write_gbs(dev)
    kernels = kernel_stats(agg, algo, pk, wr_gbs)
    total = sum(v[1] for v in agg.values())
    for name in kernels:
        kernels[name]["share"] = round(agg[name][1] / total, 4) if total else None
    dom = max(agg, key=lambda n: agg[n][1])
    kd = kernels[dom]
    if kd["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": kd["TFLOP_s"], "peak": pk["bf16_tflops_sustained"],
                "unit": "TFLOP/s"}
    elif kd["bound"] == "alu":
        roof = {"bound": "alu", "achieved": kd["TFLOP_s"], "peak": round(FP32_TFLOPS, 1),
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": kd["GB_s"], "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    # the same kernel against its HBM floor with the writes at the live
    # write-only rate where that is the longer of the two
    roof["write_aware"] = {"hbm_write_gbs_live": round(wr_gbs, 1), "floor_us": kd["hbm_floor_us"],
                           "frac": kd["hbm_floor_frac"]}
    roof["traffic"] = traffic_for(dom, args.workload)
    roof["kernel"] = dom
    roof["peak_kind"] = pk_kind
    gsum = gemm_summary(kernels, agg, algo, prof_steps, pk)

    # ---- the same step replayed from one captured CUDA graph
    graph = None
    if not args.no_graph:
        gr = moe.Graph(d, b, moe.GRAPH_LAYER_STEP, st)
        for _ in range(args.warmup):
            gr.replay(st)
        barrier(world)
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(st)
        for _ in range(args.steps):
            gr.replay(st)
        g1.record(st)
        torch.cuda.synchronize(dev)
        gms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world)
        status = moe.moe_device_status(d, b.ws, st)
        if status != moe.MOE_OK:
            raise RuntimeError(f"device status {status}: {moe.lib().moe_last_error()}")
        graph = {"ms_per_step": round(gms, 4), "value": round(world * inp.T / (gms / 1e3), 1),
                 "unit": "tokens/s", "kernels_per_step": gr.kernels,
                 "note": "moe_graph_capture(MOE_GRAPH_LAYER_STEP) replayed; same work as value"}
        gr.close()

    # ---- the weight gradients added into fp32 main gradients (gradient
    # accumulation fusion), timed on their own on the step's saved tensors: not
    # part of the step above, which stores bf16 weight gradients
    accum = None
    if not args.no_accum:
        m1 = torch.zeros(inp.E, 2 * inp.F, inp.H, dtype=torch.float32, device=dev)
        m2 = torch.zeros(inp.E, inp.H, inp.F, dtype=torch.float32, device=dev)

        def accum_call():
            moe.moe_expert_ffn_bwd_wgrad_accum(d, b.x_perm, b.h, b.d_o, b.da, b.off, m1, m2,
                                               b.ws, st)
        for _ in range(args.warmup):
            accum_call()
        torch.cuda.synchronize(dev)
        moe.moe_profile_start(2 * prof_steps + 8)
        for _ in range(prof_steps):
            accum_call()
        torch.cuda.synchronize(dev)
        aagg = _agg(moe.moe_profile_stop(2 * prof_steps + 8))
        status = moe.moe_device_status(d, b.ws, st)
        if status != moe.MOE_OK:
            raise RuntimeError(f"device status {status}: {moe.lib().moe_last_error()}")
        accum = kernel_stats(aagg, accum_algorithmic(shape), pk, wr_gbs)
        del m1, m2

    # ---- end to end through the host-buffer C-ABI calls: every step copies
    # its x and dy in from pinned host memory and its y and dx out. The
    # pipelined call runs the K steps in one call (the copies of one step
    # beside the computation of its neighbours), the per-call figure one call
    # per step.
    hx = inp.x.clone().pin_memory()
    hdy = inp.dy.clone().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    moe.moe_layer_step_host(d, b, hx, hdy, hy, hdx, st)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        moe.moe_layer_step_host(d, b, hx, hdy, hy, hdx, st)
    e2e_call_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world)
    # the second buffer set shares everything but x, dy, y and dx
    b2 = moe.LayerBuffers(d, dev, weights=b)
    for name in ("logits", "idx", "gates", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off",
                 "x_perm", "a", "h", "o", "d_o", "dgates", "da", "dx_perm", "dx32", "dw_r", "dw1",
                 "dw2", "ws"):
        setattr(b2, name, getattr(b, name))
    nh = 4  # distinct pinned host buffers, used in turn
    hxs = [inp.x.clone().pin_memory() for _ in range(nh)]
    hdys = [inp.dy.clone().pin_memory() for _ in range(nh)]
    hys = [torch.empty_like(hx).pin_memory() for _ in range(nh)]
    hdxs = [torch.empty_like(hx).pin_memory() for _ in range(nh)]
    pick = lambda ts, n: [ts[i % nh] for i in range(n)]  # noqa: E731
    moe.moe_layer_steps_host(d, b, b2, pick(hxs, 2), pick(hdys, 2), pick(hys, 2), pick(hdxs, 2),
                             st)
    barrier(world)
    t0 = time.perf_counter()
    moe.moe_layer_steps_host(d, b, b2, pick(hxs, args.steps), pick(hdys, args.steps),
                             pick(hys, args.steps), pick(hdxs, args.steps), st)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world)
    status = moe.moe_device_status(d, b.ws, st)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status {status}: {moe.lib().moe_last_error()}")
    nbytes = inp.T * inp.H * 2
    del b, b2, hxs, hdys, hys, hdxs
    torch.cuda.empty_cache()

    # ---- the other workloads of the layer: skewed routing, the emulated EP=8
    # layout, and the two-micro-batch schedule (rank 0 of a single-GPU run)
    others = {}
    if rank == 0 and world == 1 and not args.no_configs:
        sub = max(20, args.steps // 2)
        others["c3_skewed"] = measure_workload(moe, "qwen3_30b_a3b_skewed", args, dev, st, pk,
                                               wr_gbs, sub)
        others["c3_expert_buckets"] = measure_expert_buckets(
            moe, args, dev, st, pk, wr_gbs, others["c3_skewed"]["experts_by_rows"])
        others["c4_ep8"] = measure_workload(moe, "ep8_emulated", args, dev, st, pk, wr_gbs, sub)
        others["c5_schedule"] = measure_schedule(moe, args, dev, sub)

    out = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded moe_synth inputs; random-init weights of the layer's shape)",
        "config": {"workload": args.workload, **shape, "steps_per_call": "fwd+dgrad+wgrad",
                   "l2": "inputs larger than L2: %.2f GB of expert weights and %.2f GB of "
                         "activations streamed per step" % (
                             inp.E * 3 * inp.F * inp.H * 2 / 1e9,
                             inp.T * inp.k * (4 * inp.H + 6 * inp.F) * 2 / 1e9),
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(world * inp.T / e2e_s, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * nbytes, "d2h_bytes_per_step": 2 * nbytes,
                "api": "moe_layer_steps_host (K steps in one call, copies pipelined)",
                "per_call": {"value": round(world * inp.T / e2e_call_s, 1), "unit": "tokens/s",
                             "api": "moe_layer_step_host, one call per step"}},
        "gpu_launches": int(launches),
        "roofline": roof,
        "clocks": clk,
        **gsum,
        "kernels": kernels,
    }
    if sustained is not None:
        out["sustained"] = sustained
    if graph is not None:
        out["graph_step"] = graph
    if accum is not None:
        out["wgrad_accum_fp32"] = {"note": "weight gradients added into fp32 main gradients, "
                                           "timed separately; not in value",
                                   "kernels": accum}
    out.update(others)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        Ts = args.cpu_sample_tokens
        cores = cpu_cores()
        allc = oracle_timing(args.workload, Ts, cores)
        one = oracle_timing(args.workload, Ts, 1)
        out["cpu_baseline"] = {
            "value": allc["tokens_per_s"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"first {Ts} tokens of the workload, one fwd+bwd, numpy float64 + BLAS, "
                      f"{allc['seconds']} s on {cores} threads",
            "one_thread": one}
        if not args.no_configs:
            # the other workloads' oracle, all threads: the small one whole, the
            # others on the same token prefix (the two-micro-batch workload is
            # two of the balanced layer, so its rate per token is the one above)
            per = {}
            for wl in ("tiny", "qwen3_30b_a3b_skewed", "ep8_emulated"):
                import moe_synth
                n = min(Ts, moe_synth.WORKLOADS[wl]["T"])
                per[wl] = {**oracle_timing(wl, n, cores), "sample_tokens": n}
            out["cpu_baseline"]["other_workloads"] = per
    if rank == 0:
        emit(out)


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on a bounded token sample per step."""
    if rank != 0:
        return
    import moe_synth
    from oracle import moe_oracle as O
    Ts = args.ref_sample_tokens
    inp = moe_synth.workload(args.workload, T=Ts)
    # the workload's own shape: each timed step is a bounded sample of its tokens
    full_shape = dict(inp.shape_dict(), T=moe_synth.WORKLOADS[args.workload]["T"])

    def step():
        fwd = O.layer_forward(inp)
        O.layer_backward(inp, fwd)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = Ts / dt
    emit({"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s",
          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": {"workload": args.workload, **full_shape, "steps_per_call": "fwd+dgrad+wgrad",
                     "parallelism": "single process on the host cores",
                     "sample_tokens_per_step": Ts},
          "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cpu_cores(),
                           "kind": "oracle",
                           "sample": f"first {Ts} tokens of the workload per step"},
          "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


# ----------------------------------------------------------------------------- schedule
def run_schedule(args):
    """Only the two-micro-batch schedule (serial vs overlap), as its own line."""
    import combine_router_softmax_top_gb300 as moe
    from combine_router_softmax_top_gb300 import build

    build.build()
    dev = torch.device("cuda", 0)
    out = measure_schedule(moe, args, dev, args.steps)
    emit({"metric": "two-micro-batch MoE layer step, serial vs two-stream overlap", "unit": "ms",
          "higher_is_better": False, "warmup": args.warmup, **out})


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_30b_a3b_balanced")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the timing of the step replayed from a CUDA graph")
    ap.add_argument("--no-accum", action="store_true",
                    help="skip the separate timing of the fp32-accumulating weight gradients")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the skewed, EP=8 and two-micro-batch workloads")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the one-second sustained run with its own clock record")
    ap.add_argument("--cpu-sample-tokens", type=int, default=256)
    ap.add_argument("--ref-sample-tokens", type=int, default=64)
    ap.add_argument("--schedule", action="store_true",
                    help="time only the two-micro-batch scheduler (serial vs overlap)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps, always
    rank, world, local = dist_setup()
    if args.schedule:
        run_schedule(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
