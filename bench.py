#!/usr/bin/env python
"""Benchmark of the F^H D / Q gather on GB300.

Headline: F^H D voxel-sample pairs per second on the 128^3-voxel, 3D-radial
workload (M = 262,144 samples, 2,097,152 voxels), one call per step (cmpMu +
tile staging + phase + trig + complex multiply-accumulate + epilogue).  The
workload's voxels form a 128^3 grid, so the headline call is mri_fhd_grid
(the lattice-factored gather as a complex matrix product on the tensor
cores); ``--general`` times mri_fhd (per-pair phase and trig) instead.  The
same JSON line also carries the other rows of the hot path measured the same
way: both entry points with both trig paths, Q on the 128^3 stack-of-spirals
trajectory (M = 1,048,576), batched F^H D with 8 coils (M = 524,288) and the
forward model D = F rho.  ``--forward`` times the forward model as the step
(a profiling aid).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs its own 128^3 voxel slab of a stacked
volume against the same trajectory (independent problems, no collective on
the data path); the timing is the maximum over ranks.  ``--impl reference``
times the fp64 CPU oracle on the host cores instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from non_cartesian_mri_gb300 import workloads as wl  # noqa: E402

HEADLINE = "fhd_128_radial"
METRIC = "F^H D voxel-sample pairs/sec (G/s) and % of SFU/FP32 roofline, 1xGB300"
UNIT = "Gpairs/s"
L2_FLUSH_BYTES = 256 << 20

# Algorithmic operations per unit of work (the method's own minimum).
# General gather: the phase is 1 FMUL + 2 FFMA, the complex multiply-accumulate
# 4 FFMA (Q: 2), and sin + cos are two SFU (MUFU) operations.  Batched: per
# pair-coil.  Grid gather: one complex multiply-accumulate of a tabulated
# x factor and a tabulated Mu * (y, z) factor, 4 FFMA; the tables' sin/cos
# (1/R + 1/nx per pair) are excluded like the general path's range
# reduction.
ALGO_OPS = {
    "fhd": {"mufu": 2.0, "fp32": 7.0, "unit": "pair"},
    "q": {"mufu": 2.0, "fp32": 5.0, "unit": "pair"},
    "fhd_batched": {"mufu": 2.0 / 8, "fp32": 3.0 / 8 + 4.0, "unit": "pair-coil"},
    # batched on the tensor cores (groups of 3-8 coils): the complex
    # multiply-accumulate is a tensor-core product (8 flops per pair-coil,
    # 3 f16 passes each: far from binding), the phase and the sin/cos of a
    # pair stay on the SM, shared by the 8 coils of a group
    "fhd_batched_tc": {"mufu": 2.0 / 8, "fp32": 3.0 / 8, "unit": "pair-coil"},
    "grid": {"mufu": 0.0, "fp32": 4.0, "unit": "pair"},
}
# The accurate paths evaluate sin and cos in software (the MUFU's ~2^-21
# absolute error is too coarse): the exact reduction to a half turn (3 FADD),
# f^2, the odd and even polynomials (4 + 4 FFMA) and f * P: 13 FP32-pipe
# operations per sin/cos pair (the sign flip by the half turn's parity runs
# on the integer pipe).  A path that evaluates all its trig that way is bound
# by the FP32 pipe with those operations counted: that is its roofline
# ("frac"); its fraction of the SFU roofline of the fast path is reported
# beside it ("frac_vs_sfu_roofline").  A fast path whose kernel gives a share
# of its voxels the polynomial (mri_plan.fast_fp32_voxels) is charged that
# share on the FP32 pipe (plus the multiply turning radians into half turns)
# and the rest on the SFU.
TRIG_FP32_OPS = 13.0
TRIG_FP32_OPS_FROM_RADIANS = TRIG_FP32_OPS + 1.0
# The tensor-core grid kernels: one complex multiply-accumulate is
# 8 real flops per pair; each fp32-accurate product takes three f16 MMA
# passes (hi*hi + hi*lo + lo*hi), so its peak is the dense f16 peak / 3, and
# dense f16 runs at the measured bf16 rate.
TC_FLOPS_PER_PAIR = 8.0
TC_PASSES = 3.0
F16_PER_BF16 = 1.0
# Per-SM-per-clock rates of sm_103a, measured live by the mri_microbench
# probes (one CTA of 1024 threads per SM): FP32 128 lanes (scalar FFMA, and
# FFMA2, whose packed pairs hold the pipe for two cycles), MUFU sin / cos 16.
NOMINAL = {"mufu": 16.0, "fp32": 128.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--trig", choices=["fast", "accurate", "fast_rr"], default="fast")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--grid-edge", type=int, default=None,
                    help="override the voxel-grid edge L (smaller cases for profiling)")
    ap.add_argument("--general", action="store_true",
                    help="time F^H D / Q through mri_fhd / mri_q instead of the grid entry points")
    ap.add_argument("--no-paths", action="store_true",
                    help="skip the accurate/Q/batched sub-measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--forward", action="store_true",
                    help="time the forward model D = F rho (of a seeded image) on the "
                         "workload's trajectory and grid instead of F^H D (profiling aid; "
                         "implies --no-paths --no-e2e)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--find-rho", action="store_true",
                    help="also measure the find-rho step (Toeplitz product, CG iteration) and "
                         "the gridding reconstruction when the other paths are skipped")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# process group (one rank per GPU under torchrun)
# ---------------------------------------------------------------------------

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, world, rank, device):
        self.world, self.rank = world, rank
        self.pg = None
        if world > 1:
            import torch.distributed as td
            backend = "nccl" if device.type == "cuda" else "gloo"
            td.init_process_group(backend=backend, world_size=world, rank=rank)
            self.td = td

    def barrier(self):
        if self.world > 1:
            self.td.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.td.destroy_process_group()


def slab(w: wl.Workload, rank: int) -> wl.Workload:
    """Rank r's problem: the same trajectory against the voxel slab z + r*L."""
    if rank == 0:
        return w
    z = (w.z + np.float32(rank * w.L)).astype(np.float32)
    return wl.Workload(w.name, w.kind, w.L, w.kx, w.ky, w.kz, w.x, w.y, z, w.rPhi, w.iPhi,
                       w.rD, w.iD, w.B, dict(w.meta, slab=rank))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.fh = None

    def __enter__(self):
        try:
            self.fh = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.fh is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.fh.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.fh.read())) if len(r) >= 9]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def to_dev(w: wl.Workload, torch):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    out = {k: d(getattr(w, k)) for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi", "iPhi")}
    if w.rD is not None:
        out["rD"] = d(w.rD)
        out["iD"] = d(w.iD)
    out["xs"], out["ys"], out["zs"] = (d(a) for a in w.axes())
    return out


def call(mri, kind, t, trig, out=None, grid=False):
    if grid and kind == "fhd_batched":
        return mri.fhd_batched_grid(t["kx"], t["ky"], t["kz"], t["xs"], t["ys"], t["zs"],
                                    t["rPhi"], t["iPhi"], t["rD"], t["iD"], trig=trig, out=out)
    if grid and kind == "fhd":
        return mri.fhd_grid(t["kx"], t["ky"], t["kz"], t["xs"], t["ys"], t["zs"], t["rPhi"],
                            t["iPhi"], t["rD"], t["iD"], trig=trig, out=out)
    if grid and kind == "q":
        return mri.q_grid(t["kx"], t["ky"], t["kz"], t["xs"], t["ys"], t["zs"], t["rPhi"],
                          t["iPhi"], trig=trig, out=out)
    if kind == "fhd":
        return mri.fhd(t["kx"], t["ky"], t["kz"], t["x"], t["y"], t["z"], t["rPhi"], t["iPhi"],
                       t["rD"], t["iD"], trig=trig, out=out)
    if kind == "q":
        return mri.q(t["kx"], t["ky"], t["kz"], t["x"], t["y"], t["z"], t["rPhi"], t["iPhi"],
                     trig=trig, out=out)
    return mri.fhd_batched(t["kx"], t["ky"], t["kz"], t["x"], t["y"], t["z"], t["rPhi"],
                           t["iPhi"], t["rD"], t["iD"], trig=trig, out=out)


ENTRY = {("fhd", True): "mri_fhd_grid", ("q", True): "mri_q_grid",
         ("fhd_batched", True): "mri_fhd_batched_grid",
         ("fhd", False): "mri_fhd", ("q", False): "mri_q",
         ("fhd_batched", False): "mri_fhd_batched"}


def grid_or_general_plan(mri, w, grid):
    if grid and w.kind == "fhd_batched":
        return mri.plan_grid_batched(w.B, w.M, w.L, w.L, w.L)
    if grid:
        return mri.plan_grid(w.kind, w.M, w.L, w.L, w.L)
    return mri.plan(w.kind, w.M, w.N, B=w.B)


def timed_steps(torch, mri, dist, fn, steps, warmup, flush):
    """W untimed steps, then K steps bracketed by barrier + synchronize; each
    step's device time from CUDA events on the launching stream, the L2
    flushed (256 MiB write) before every step outside the events."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    wall0 = time.perf_counter()
    with mri.gather_timing() as gt:
        for k in range(steps):
            flush()
            evs[k][0].record(stream)
            fn()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    step_ms = [a.elapsed_time(b) for a, b in evs]
    return {"step_ms": step_ms, "gather_ms": gt.ms, "gather_launches": gt.launches,
            "wall_s": wall}


def unit_rates(mri):
    r = {}
    for probe in ("sin", "cos", "ffma", "ffma2"):
        mri.microbench(probe, ctas_per_sm=1, threads=1024, iters=1 << 10)
        r[probe] = round(mri.microbench(probe, ctas_per_sm=1, threads=1024,
                                        iters=1 << 13)["per_sm_per_clk"], 2)
    return r


def algo_ops(kind, trig="fast", fp32_share=0.0):
    """Operations per work unit.  trig = "accurate" (or "accurate_fp32"): every
    sin/cos pair is software trig on the FP32 pipe; a fast path with
    fp32_share > 0 moves that share of its sin/cos pairs there."""
    ops = dict(ALGO_OPS[kind])
    pairs = ops["mufu"] / 2.0                  # sin/cos pairs per work unit
    if trig in ("accurate", "accurate_fp32") and pairs:
        ops["fp32"] += TRIG_FP32_OPS * pairs
        ops["mufu"] = 0.0
    elif trig == "fast" and fp32_share > 0 and pairs:
        ops["fp32"] += TRIG_FP32_OPS_FROM_RADIANS * pairs * fp32_share
        ops["mufu"] *= 1.0 - fp32_share
    return ops


def peak_per_sm_clk(kind, rates, trig="fast", fp32_share=0.0):
    """Binding roofline in work units per SM per clock: min over the two units."""
    ops = algo_ops(kind, trig, fp32_share)
    mufu = NOMINAL["mufu"] if rates is None else min(rates["sin"], rates["cos"])
    fp32 = NOMINAL["fp32"] if rates is None else rates["ffma"]
    # nominal integers when the probe agrees within 10%
    if abs(mufu - NOMINAL["mufu"]) <= 0.1 * NOMINAL["mufu"]:
        mufu = NOMINAL["mufu"]
    if abs(fp32 - NOMINAL["fp32"]) <= 0.1 * NOMINAL["fp32"]:
        fp32 = NOMINAL["fp32"]
    by_mufu = mufu / ops["mufu"] if ops["mufu"] else float("inf")
    by_fp32 = fp32 / ops["fp32"]
    return min(by_mufu, by_fp32), ("mufu" if by_mufu <= by_fp32 else "fp32"), mufu, fp32


# The sources a kernel's DRAM traffic depends on (its code and the host code
# that plans its launch); a stored traffic figure is valid while they are
# unchanged.
_COMMON_SOURCES = ("ptx.cuh", "gather.cuh", "sincospi_coeffs.h", "mri_abi.cu")
TRAFFIC_SOURCES = {
    "grid_tc": _COMMON_SOURCES + ("gather_grid.cuh", "gather_grid_tc.cuh",
                                  "gather_grid_tc_ws.cuh", "kernels_grid_tc.cu"),
    "grid_tc_fwd": _COMMON_SOURCES + ("gather_grid.cuh", "gather_grid_tc.cuh",
                                      "gather_grid_tc_fwd.cuh", "kernels_grid_tc.cu"),
    "toeplitz": ("fft.cuh", "kernels_toeplitz.cu"),
    "gridding": ("fft.cuh", "kernels_gridding.cu"),
    # the general gather on pairs of floats (F^H D, Q, the forward model)
    "pair": ("ptx.cuh", "gather.cuh", "gather_pair.cuh", "sincospi_coeffs.h",
             "kernels_single.cu", "mri_abi.cu"),
    # the batched general gather on the tensor cores
    "coils_tc": _COMMON_SOURCES + ("gather_grid.cuh", "gather_grid_tc.cuh",
                                   "gather_coils_tc.cuh", "kernels_coils_tc.cu"),
}


def gather_source_hash(kind="grid_tc"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "non_cartesian_mri_gb300", "csrc")
    names = TRAFFIC_SOURCES.get(kind)
    if names is None:   # any other kernel: every source
        names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind, trig, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    trig path and workload, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = rec.get(f"{kind}:{workload}:{trig}")
    if not entry or entry.get("source_hash") != gather_source_hash(kind):
        return None
    return entry.get("dram_bytes_per_launch")


def roofline_tensor(w, res, peaks, trig, units):
    per_launch = res["gather_ms"] / max(res["gather_launches"], 1) / 1e3
    launches_per_step = res["gather_launches"] / len(res["step_ms"])
    pairs_s = units / launches_per_step / per_launch
    achieved = pairs_s * TC_FLOPS_PER_PAIR / 1e12
    bf16 = float(peaks.get("bf16_tflops", 1900.0))
    peak = bf16 * F16_PER_BF16 / TC_PASSES
    return {"bound": "tensor", "binding_unit": "tcgen05 kind::f16 (f16 x f16 -> f32)",
            "achieved": round(achieved, 2),
            "peak": round(peak, 2), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic("grid_tc", trig, w.name),
            "peak_basis": (f"bf16 burst {bf16:g} TFLOP/s ({'measured, MEASURED_PEAKS.json' if 'bf16_tflops' in peaks else 'recipe fallback'})"
                           f" = dense f16 rate, / {TC_PASSES:g} f16 products per fp32 product;"
                           f" algorithmic {TC_FLOPS_PER_PAIR:g} flops per voxel-sample pair"),
            "executed_tflops": round(achieved * TC_PASSES, 2),
            "pairs_per_s": round(pairs_s / 1e9, 2),
            "unit_pairs": "Gpair-coils/s" if w.B > 1 else "Gpairs/s",
            "gather_ms_per_launch": round(per_launch * 1e3, 3)}


def roofline(kind, w, res, rates, sms, sm_max_mhz, sm_mhz, trig, grid=False, plan=None,
             peaks=None):
    if grid and plan and plan.get("tensor_cores"):
        return roofline_tensor(w, res, peaks or {}, trig,
                               w.pairs * (w.B if kind == "fhd_batched" else 1))
    units = w.pairs * (w.B if kind == "fhd_batched" else 1)
    akind = "grid" if grid else kind
    if kind == "fhd_batched" and not grid and plan and plan.get("tensor_cores"):
        akind = "fhd_batched_tc"
    per_launch = res["gather_ms"] / max(res["gather_launches"], 1) / 1e3
    launches_per_step = res["gather_launches"] / len(res["step_ms"])
    achieved = units / launches_per_step / per_launch / 1e9
    share = 0.0
    if trig == "fast" and not grid and plan and plan.get("voxels_per_thread"):
        share = plan.get("fast_fp32_voxels", 0) / plan["voxels_per_thread"]
    per_clk, unit, mufu, fp32 = peak_per_sm_clk(akind, rates, trig, share)
    peak = per_clk * sms * sm_max_mhz * 1e6 / 1e9
    ops = algo_ops(akind, trig, share)
    basis = (f"{sms} SMs x {sm_max_mhz:.0f} MHz x min(MUFU {mufu:g}/{ops['mufu']:g}, "
             f"FP32 {fp32:g}/{ops['fp32']:g}) per SM-clock") if ops["mufu"] else (
             f"{sms} SMs x {sm_max_mhz:.0f} MHz x FP32 {fp32:g}/{ops['fp32']:g} per SM-clock")
    if share:
        basis += (f"; {share:.3g} of the voxels take the polynomial on the FP32 pipe "
                  f"({TRIG_FP32_OPS_FROM_RADIANS:g} ops per sin/cos pair)")
    if trig == "accurate" and ALGO_OPS[akind]["mufu"]:
        basis += f" ({TRIG_FP32_OPS:g} FP32 ops per software sin/cos pair counted)"
    out = {"bound": "alu", "binding_unit": unit, "achieved": round(achieved, 2),
           "peak": round(peak, 2),
           "unit": "G" + ops["unit"] + "s/s",
           "frac": round(achieved / peak, 4),
           "traffic": profiled_traffic(akind if grid else
                                       ("pair" if kind in ("fhd", "q") else
                                        "coils_tc" if akind == "fhd_batched_tc" else kind),
                                       trig, w.name),
           "peak_basis": basis,
           "gather_ms_per_launch": round(per_launch * 1e3, 3)}
    if sm_mhz:
        out["frac_at_sampled_clock"] = round(achieved / (per_clk * sms * sm_mhz * 1e-3), 4)
        out["units_per_sm_clk"] = round(achieved * 1e9 / (sms * sm_mhz * 1e6), 3)
    if ALGO_OPS[akind]["mufu"] and (trig == "accurate" or share):
        # the fast path's roofline with every sin/cos on the SFU, for comparison
        sper, _, _, _ = peak_per_sm_clk(akind, rates, "fast", 0.0)
        out["frac_vs_sfu_roofline"] = round(achieved / (sper * sms * sm_max_mhz * 1e-3), 4)
    return out


def cpu_baseline(w: wl.Workload, target_s: float = 12.0):
    """The oracle, as it stands, on a seeded voxel sample of the workload."""
    import oracle
    cores = oracle.threads(0)
    probe = wl.voxel_subset(w.N, 32, 9)
    t0 = time.perf_counter()
    oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    count = int(min(max(32 * target_s / dt, 64), 65536, w.N))
    idx = wl.voxel_subset(w.N, count, 10)
    t0 = time.perf_counter()
    oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx)
    dt = time.perf_counter() - t0
    pairs = count * w.M
    # the same oracle on one core, on a smaller sample (about 2 s)
    count1 = int(min(max(32 * 2.0 / (dt / count * cores * 32), 16), count))
    idx1 = wl.voxel_subset(w.N, count1, 11)
    t0 = time.perf_counter()
    oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx1, threads=1)
    dt1 = time.perf_counter() - t0
    return {"value": round(pairs / dt / 1e9, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{count} seeded voxels x all {w.M} samples of {w.name} "
                      f"({pairs:.3g} pairs, {dt:.1f} s, fp64, OpenMP over voxels)",
            "one_core": {"value": round(count1 * w.M / dt1 / 1e9, 5), "unit": UNIT,
                         "sample": f"{count1} seeded voxels x all {w.M} samples, {dt1:.1f} s"}}


def e2e(torch, mri, dist, w, trig, steps, warmup, grid=False):
    """Public API with pinned host buffers: H2D of the inputs, the call, D2H of
    the outputs, all inside the timed region."""
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    k = [pin(getattr(w, n)) for n in ("kx", "ky", "kz")]
    wts = [pin(getattr(w, n)) for n in ("rPhi", "iPhi", "rD", "iD")]
    vox = [pin(a) for a in w.axes()] if grid else [pin(getattr(w, n)) for n in ("x", "y", "z")]
    host = k + vox + wts
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = 2 * w.N * 4

    def step():
        f = mri.fhd_grid if grid else mri.fhd
        return f(*k, *vox, *wts, trig=trig)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    dist.barrier()
    mean_s = dist.max(statistics.mean(times))
    return {"value": round(w.pairs * dist.world / mean_s / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(mean_s * 1e3, 3)}


# The find-rho step (CG on (F^H F + lambda I) x = F^H D with the Toeplitz
# product): HBM-bound.  Bytes per product for N voxels, stage by stage (the
# work array holds half the doubled grid, 4N complex values of 8 bytes; the
# real spectrum K the whole doubled grid, 8N floats):
#   x forward   read v (8N), write 2N values (16N)
#   y forward   read 2N values (16N), write 4N (32N)
#   z           read 4N (32N) and K (32N), write 4N (32N)
#   y inverse   read 4N (32N), write 2N (16N)
#   x inverse   read 2N (16N) and v (8N), write the result (8N)
# = 248 bytes per voxel.  The compulsory part (v, K and the result once) is
# 48.  A CG iteration adds the x / r update (48N) and, inside the first
# stage, the direction update p = r + beta p (r read, p written: 16N); p.Ap
# is summed inside the last stage.
TOEPLITZ_BYTES_PER_VOXEL = 8 + 16 + 16 + 32 + 32 + 32 + 32 + 32 + 16 + 16 + 8 + 8
TOEPLITZ_COMPULSORY_BYTES_PER_VOXEL = 8 + 32 + 8
CG_EXTRA_BYTES_PER_VOXEL = 48 + 16


def find_rho(torch, mri, dist, args, flush, peaks):
    """Toeplitz product and CG iteration on the headline trajectory and grid."""
    w = wl.make_workload(HEADLINE)
    t = to_dev(w, torch)
    shape = (w.L, w.L, w.L)
    K = mri.toeplitz_kernel(t["kx"], t["ky"], t["kz"], t["rPhi"], t["iPhi"], shape,
                            trig=args.trig)
    rng = np.random.default_rng(77)
    v = [torch.from_numpy(rng.standard_normal(w.N).astype(np.float32)).cuda() for _ in range(2)]
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    out = {"workload": f"{w.name} trajectory, {w.L}^3 grid (doubled grid {2 * w.L}^3)",
           "trig_of_q": args.trig}
    iters = 10
    for name, fn, per_step, bpv in (
            ("toeplitz_apply", lambda: mri.toeplitz_apply(K, v[0], v[1], lam=0.01), 1,
             TOEPLITZ_BYTES_PER_VOXEL),
            ("cg_iteration", lambda: mri.cg_solve(K, v[0], v[1], lam=0.01, iters=iters), iters,
             TOEPLITZ_BYTES_PER_VOXEL + CG_EXTRA_BYTES_PER_VOXEL)):
        res = timed_steps(torch, mri, dist, fn, args.steps, args.warmup, flush)
        ms = statistics.mean(res["step_ms"]) / per_step
        achieved = bpv * w.N / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "value": round(w.N / (ms * 1e-3) / 1e9, 3),
                     "unit": "Gvoxels/s",
                     "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                                  "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                                  "traffic": profiled_traffic(
                                      "toeplitz",
                                      "product" if name == "toeplitz_apply" else "cg_iteration",
                                      w.name),
                                  "algorithmic_bytes_per_voxel": bpv,
                                  "compulsory_bytes_per_voxel":
                                      TOEPLITZ_COMPULSORY_BYTES_PER_VOXEL}}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    mri.toeplitz_kernel(t["kx"], t["ky"], t["kz"], t["rPhi"], t["iPhi"], shape, trig=args.trig)
    t1.record()
    torch.cuda.synchronize()
    out["toeplitz_kernel_ms_once"] = round(t0.elapsed_time(t1), 2)
    del t, K, v
    torch.cuda.empty_cache()
    if dist.rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_toeplitz(w)
    return out


def cpu_baseline_toeplitz(w):
    """The oracle's Toeplitz product (oracle.toeplitz.fhf_fft: numpy FFTs of
    the doubled grid, fp64), as it stands, once on the workload's grid.  Its
    cost does not depend on the values, so a seeded Q grid of the right shape
    stands in for the trajectory's (whose oracle evaluation would take hours)."""
    from oracle import toeplitz as T
    rng = np.random.default_rng(78)
    L = w.L
    Qc = rng.standard_normal((2 * L,) * 3) + 1j * rng.standard_normal((2 * L,) * 3)
    rho = rng.standard_normal((L,) * 3) + 1j * rng.standard_normal((L,) * 3)
    t0 = time.perf_counter()
    T.fhf_fft(Qc, rho)
    dt = time.perf_counter() - t0
    return {"value": round(w.N / dt / 1e9, 5), "unit": "Gvoxels/s", "cores": 1,
            "kind": "oracle",
            "sample": f"one product on the {L}^3 grid ({2 * L}^3 numpy FFTs, fp64, one "
                      f"thread), {dt:.1f} s"}


# The gridding reconstruction: bytes per call for M samples on N voxels --
# the samples read once (k 12, Phi 8, D 8 = 28 B), the grid zeroed (8 B per
# voxel), the 8M atomic adds (into L2: the grid of a 128^3 image is 16 MB),
# the inverse FFT's three passes (16 B per voxel each), the signs pass (8 B
# in, 8 B out).  Algorithmic HBM bytes: 28 M + 72 N.
GRIDDING_BYTES_PER_SAMPLE = 28
GRIDDING_BYTES_PER_VOXEL = 8 + 3 * 16 + 16


def gridding(torch, mri, dist, args, flush, peaks):
    """The gridding reconstruction on the headline trajectory and grid."""
    w = wl.make_workload(HEADLINE)
    t = to_dev(w, torch)
    shape = (w.L, w.L, w.L)
    fn = lambda: mri.gridding(t["kx"], t["ky"], t["kz"], t["rPhi"], t["iPhi"], t["rD"],  # noqa: E731
                              t["iD"], shape)
    res = timed_steps(torch, mri, dist, fn, args.steps, args.warmup, flush)
    ms = statistics.mean(res["step_ms"])
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    nbytes = GRIDDING_BYTES_PER_SAMPLE * w.M + GRIDDING_BYTES_PER_VOXEL * w.N
    achieved = nbytes / (ms * 1e-3) / 1e9
    del t
    torch.cuda.empty_cache()
    out = {"workload": f"{w.name}: M={w.M:,} samples onto a {w.L}^3 grid",
           "ms": round(ms, 4), "value": round(w.M / (ms * 1e-3) / 1e9, 3),
           "unit": "Gsamples/s",
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                        "unit": "GB/s", "frac": round(achieved / hbm, 4),
                        "traffic": profiled_traffic("gridding", "call", w.name),
                        "algorithmic_bytes": nbytes}}
    if dist.rank == 0 and not args.no_cpu:
        from oracle import gridding as Gr
        t0 = time.perf_counter()
        Gr.gridding_recon(w.kx, w.ky, w.kz, w.rPhi, w.iPhi, w.rD, w.iD, shape)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": round(w.M / dt / 1e9, 5), "unit": "Gsamples/s",
                               "cores": 1, "kind": "oracle",
                               "sample": f"the whole reconstruction once (numpy, fp64, one "
                                         f"thread), {dt:.1f} s"}
    return out


def run_ours(args):
    import torch
    import non_cartesian_mri_gb300 as mri
    from non_cartesian_mri_gb300 import build

    world, rank, local = dist_info()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    build.build()
    mri.load()
    dist = Dist(world, rank, torch.device("cuda", local))
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peaks = json.load(fh)
    except (OSError, ValueError):
        pass
    sm_max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_ctr = [0]

    def flush():
        flush_ctr[0] += 1
        flush_buf.fill_(float(flush_ctr[0] & 7))

    rates = unit_rates(mri)

    w = slab(wl.make_workload(args.workload, L=args.grid_edge), rank)
    kind = w.kind
    t = to_dev(w, torch)
    out = (torch.empty((w.B, w.N) if kind == "fhd_batched" else (w.N,), device="cuda"),
           torch.empty((w.B, w.N) if kind == "fhd_batched" else (w.N,), device="cuda"))
    grid = not args.general
    if args.forward:
        # the forward model D = F rho of a seeded complex image
        args.no_paths = args.no_e2e = True
        rng = np.random.default_rng(1000 + w.meta.get("seed", 0))
        rho = [torch.from_numpy(rng.standard_normal(w.N).astype(np.float32)).cuda()
               for _ in range(2)]
        if grid:
            step = lambda: mri.forward_grid(t["kx"], t["ky"], t["kz"], t["xs"], t["ys"],  # noqa: E731
                                            t["zs"], rho[0], rho[1], trig=args.trig)
            plan = {"launches": 4, "tensor_cores": 1, "samples_per_tile": 128}
        else:
            step = lambda: mri.forward(t["kx"], t["ky"], t["kz"], t["x"], t["y"], t["z"],  # noqa: E731
                                       rho[0], rho[1], trig=args.trig)
            plan = mri.plan("fhd", w.N, w.M)
    else:
        step = lambda: call(mri, kind, t, args.trig, out, grid)  # noqa: E731
        plan = grid_or_general_plan(mri, w, grid)
    with ClockSampler(local) as clk:
        res = timed_steps(torch, mri, dist, step, args.steps, args.warmup, flush)
    clocks = clk.summary()
    mean_s = dist.max(statistics.mean(res["step_ms"]) / 1e3)
    units = w.pairs * (w.B if kind == "fhd_batched" else 1)
    value = units * world / mean_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded generators, no dataset)",
        "config": {"workload": f"{w.name}: {wl.WORKLOADS[w.name]}", "voxels": w.N,
                   "samples": w.M, "coils": w.B, "trig": args.trig,
                   "entry": (("mri_forward_grid" if grid else "mri_forward") if args.forward
                             else ENTRY[(kind, grid)]),
                   "l2": "flushed before every step (256 MiB write, outside the step events)",
                   "parallelism": "one independent voxel slab per rank" if world > 1
                   else "single GPU",
                   "plan": plan},
        "roofline": roofline(kind, w, res, rates, sms, sm_max_mhz, clocks.get("sm_mhz"),
                             args.trig, grid, plan, peaks),
        "gpu_launches": plan["launches"] * args.steps,
        "clocks": clocks,
        "unit_rates_per_sm_clk": rates,
    }
    line["roofline"]["sm_max_mhz_basis"] = "MEASURED_PEAKS.json sm_max_mhz" if peaks else "recipe"
    if args.forward:
        line["config"]["workload"] += " (forward model of a seeded complex image)"
        line["roofline"]["traffic"] = profiled_traffic("grid_tc_fwd" if grid else "forward",
                                                       args.trig, w.name)

    if not args.no_e2e and kind == "fhd":
        line["e2e"] = e2e(torch, mri, dist, w, args.trig, max(args.steps, 2), 1, grid)
    del t, out
    torch.cuda.empty_cache()

    if not args.no_paths and args.workload == HEADLINE and world == 1 and not args.grid_edge:
        paths = {}
        for name, wname, trig, pgrid in (
                ("fhd_grid_accurate", HEADLINE, "accurate", True),
                ("fhd_grid_fast_rr", HEADLINE, "fast_rr", True),
                ("fhd_general_fast", HEADLINE, "fast", False),
                ("fhd_general_fast_rr", HEADLINE, "fast_rr", False),
                ("fhd_general_accurate", HEADLINE, "accurate", False),
                ("fhd_64_grid_fast", "fhd_64", "fast", True),
                ("fhd_64_grid_accurate", "fhd_64", "accurate", True),
                ("fhd_64_general_fast", "fhd_64", "fast", False),
                ("fhd_64_general_accurate", "fhd_64", "accurate", False),
                ("fhd_tiny_grid_fast", "fhd_tiny", "fast", True),
                ("fhd_tiny_general_fast", "fhd_tiny", "fast", False),
                ("q_grid_fast", "q_128", "fast", True),
                ("q_grid_accurate", "q_128", "accurate", True),
                ("q_general_fast", "q_128", "fast", False),
                ("q_general_accurate", "q_128", "accurate", False),
                ("fhd_batched_grid_fast", "fhd_batched_128", "fast", True),
                ("fhd_batched_grid_accurate", "fhd_batched_128", "accurate", True),
                ("fhd_batched_fast", "fhd_batched_128", "fast", False),
                ("fhd_batched_accurate", "fhd_batched_128", "accurate", False),
                ("forward_grid_fast", HEADLINE, "fast", True),
                ("forward_grid_accurate", HEADLINE, "accurate", True),
                ("forward_general_fast", HEADLINE, "fast", False),
                ("forward_general_accurate", HEADLINE, "accurate", False)):
            if wname == HEADLINE and name.startswith("fhd_") and \
                    (name.startswith("fhd_grid") == grid) and trig == args.trig:
                continue                     # the headline itself
            pw = wl.make_workload(wname)
            pt = to_dev(pw, torch)
            po = None
            fwd = name.startswith("forward")
            if fwd:
                # the forward model D = F rho of a seeded complex image
                rng = np.random.default_rng(1000 + pw.meta.get("seed", 0))
                rho = [torch.from_numpy(rng.standard_normal(pw.N).astype(np.float32)).cuda()
                       for _ in range(2)]
                if pgrid:
                    fn = lambda: mri.forward_grid(pt["kx"], pt["ky"], pt["kz"], pt["xs"],  # noqa: E731
                                                  pt["ys"], pt["zs"], rho[0], rho[1], trig=trig)
                else:
                    fn = lambda: mri.forward(pt["kx"], pt["ky"], pt["kz"], pt["x"],  # noqa: E731
                                             pt["y"], pt["z"], rho[0], rho[1], trig=trig)
            else:
                fn = lambda: call(mri, pw.kind, pt, trig, po, pgrid)  # noqa: E731
            # slow paths (the general kernels on the largest workloads take up
            # to seconds per call) time fewer steps, at least 3, about 4 s
            flush()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            one = time.perf_counter() - t0
            psteps = max(3, min(args.steps, int(4.0 / max(one, 1e-6))))
            pres = timed_steps(torch, mri, dist, fn, psteps, max(args.warmup - 1, 2), flush)
            pm = statistics.mean(pres["step_ms"]) / 1e3
            punits = pw.pairs * (pw.B if pw.kind == "fhd_batched" else 1)
            if fwd and pgrid:
                # one prep (bound, rho table, row coordinates: 3 kernels) + the gather
                pplan = {"launches": 4, "tensor_cores": 1, "samples_per_tile": 128}
            elif fwd:
                pplan = mri.plan("fhd", pw.N, pw.M)
            else:
                pplan = grid_or_general_plan(mri, pw, pgrid)
            paths[name] = {
                "workload": f"{pw.name}: {wl.WORKLOADS[pw.name]}"
                            + (" (forward model of a seeded complex image)" if fwd else ""),
                "trig": trig,
                "entry": ("mri_forward_grid" if pgrid else "mri_forward") if fwd
                         else ENTRY[(pw.kind, pgrid)],
                "value": round(punits / pm / 1e9, 2),
                "unit": "G" + ALGO_OPS[pw.kind]["unit"] + "s/s",
                "ms_per_step": round(pm * 1e3, 3),
                "roofline": roofline(pw.kind, pw, pres, rates, sms, sm_max_mhz,
                                     clocks.get("sm_mhz"), trig, pgrid, pplan, peaks),
                "gpu_launches": pplan["launches"] * psteps,
                "steps": psteps,
            }
            if fwd:
                # the forward kernels have their own traffic records
                paths[name]["roofline"]["traffic"] = profiled_traffic(
                    "grid_tc_fwd" if pgrid else "forward", trig, pw.name)
            if pw.kind == "fhd_batched":
                paths[name]["trajectory_pairs_per_s_G"] = round(pw.pairs / pm / 1e9, 2)
            del pt
            torch.cuda.empty_cache()
        line["paths"] = paths
    if world == 1 and args.workload == HEADLINE and not args.grid_edge and not args.forward and (
            not args.no_paths or args.find_rho):
        line["find_rho"] = find_rho(torch, mri, dist, args, flush, peaks)
        line["gridding"] = gridding(torch, mri, dist, args, flush, peaks)

    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl.make_workload(args.workload, L=args.grid_edge))
    errs = mri.device_errors(clear=True)
    if errs:
        line["device_errors"] = errs
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    w = wl.make_workload(args.workload)
    cores = oracle.threads(0)
    probe = wl.voxel_subset(w.N, 16, 11)
    t0 = time.perf_counter()
    run = {"fhd": oracle.fhd, "q": oracle.q, "fhd_batched": oracle.fhd_batched}[w.kind]

    def step(idx):
        if w.kind == "q":
            run(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, idx=idx)
        else:
            run(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx)

    step(probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    per_step_s = min(150.0 / max(args.steps + args.warmup, 1), 15.0)
    count = int(min(max(16 * per_step_s / dt, 16), 65536, w.N))
    times = []
    for k in range(args.warmup + args.steps):
        idx = wl.voxel_subset(w.N, count, 1000 + k)
        t0 = time.perf_counter()
        step(idx)
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    mean_s = statistics.mean(times)
    units = count * w.M * (w.B if w.kind == "fhd_batched" else 1)
    value = units / mean_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generators, no dataset)",
        "config": {"workload": f"{w.name}: {wl.WORKLOADS[w.name]}", "voxels": w.N,
                   "samples": w.M, "coils": w.B,
                   "sample_per_step": f"{count} seeded voxels x all {w.M} samples"},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": f"{count} seeded voxels per step x all {w.M} samples "
                                   f"of {w.name}, fp64, OpenMP over voxels"},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
