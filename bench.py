#!/usr/bin/env python
"""Benchmark of the flux-differencing volume term on GB300.

One step = one evaluation of the volume term (esdg_volume_rhs) over the whole
mesh of the workload.  Default workload: the baroclinic-channel-shaped mesh,
64x16x8 warped elements of order N = 7 (4,194,304 nodes), FP64; the FP32
kernel on the same mesh is timed in the same run and reported under "fp32".
The inputs (503 MB in FP64, 252 MB in FP32) are larger than the 129 MB L2, so
no flush is needed between steps.

Metric: volume-term GDOF/s = nodes / (kernel time per step), whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank evaluates its own copy of the workload
(elements are independent, so ranks need no exchange: weak scaling); rank 0
prints one JSON line with the total over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

# ---------------------------------------------------------------------------
# algorithmic operation counts (per unit of work), counted from the formulas
# of the volume term with every +, -, *, / as one operation and a logarithm as
# one operation (fused multiply-adds count two):
#   per unordered node pair and direction, both nodes' contributions:
#     averaged metric 3, averaged velocity 3, {{u}}.n 5, log mean of rho 3,
#     inverse log mean of b 3, {{rho}} and {{b}} 2, p_hat 2, {{phi}} and [[phi]] 2,
#     {{|u|^2}} 1, |{{u}}|^2 5, rho_hat 2, gravity scalar 2 and partner scaling 2,
#     F_rho 1, momentum 9, gravity vectors 6, F_E 7, accumulation into both
#     nodes 26                                               -> 84
#   per node: u 4, |u|^2 5, p 6, b and 1/b 3, two logarithms 2, h 3,
#     1/w scaling of three directions 15                     -> 38
#   per end node of a line (2D form diagonal): 20, on 2 of the Nq nodes of
#     each line in each of the 3 directions
# Pairs per node: 3 (Nq - 1) / 2 (each unordered pair once, Sec. 4.1).
PAIR_OPS = 84
NODE_OPS = 38
DIAG_OPS = 20


def flops_per_dof(N: int, form2d: bool = True) -> float:
    Nq = N + 1
    f = PAIR_OPS * 3.0 * (Nq - 1) / 2.0 + NODE_OPS
    if form2d:
        f += DIAG_OPS * 3.0 * 2.0 / Nq
    return f


BYTES_PER_DOF = {"fp64": 20 * 8, "fp32": 20 * 4, "fp64ff": 20 * 8}  # 15 planes read + 5 written

# Surface term, algorithmic operations per face node (same counting rules),
# from the formulas of the surface kernel:
#   interior face node (evaluated once for both sides): two node states
#     (1/rho, u, |u|^2, p, b, two logarithms) 38, entropy-conserving flux
#     with gravity 69, matrix dissipation (averaged state, sound speed,
#     entropy-variable jumps, wave strengths, projections) 128, both sides'
#     fluxes 31, the physical flux subtracted on both sides (2D form) 54,
#     1/w_0 accumulation into both nodes 20                   -> 340
#   slip-wall face node: one node state 19, mirror state 24, flux 69,
#     dissipation 128, fluxes 31, physical flux 27, accumulation 10 -> 308
# Values moved per face node: interior 2 x (5 + 1 + 3) read + 2 x 5
# read-modify-written = 38; wall 9 + 5 + 5 = 19.
GAMMA = 1.4
STEP_DT = 1.0e-3  # s; stable on every workload here (timing does not depend on it)
RK_STAGE_VALUES = 26  # per node: q, rhs, dq read (5 each), J, dq and q written (5 each)

SURF_IFACE_OPS = 340
SURF_WALL_OPS = 308
SURF_IFACE_VALUES = 38
SURF_WALL_VALUES = 19


def surface_counts(cfg):
    """(interior face nodes, wall face nodes) over the three direction passes."""
    Nq2 = (cfg.N + 1) ** 2
    K = cfg.K
    Kd = (cfg.Kx, cfg.Ky, cfg.Kz)
    inner = walls = 0
    for r in range(3):
        plane = (K // Kd[r]) * Nq2
        if cfg.bc[r]:
            inner += K * Nq2 - plane
            walls += 2 * plane
        else:
            inner += K * Nq2
    return inner, walls

NOMINAL_FP64_TFLOPS = 1.25  # GB300 FP64 vector, nominal


_CSRC = os.path.join(ROOT, "flux_differencing_gb300", "csrc")
_NUMERIC = ("numeric.cuh", "floatfloat.cuh", "log_fp64.cuh", "log_table.inc", "esdg_internal.h", "surface_flux.cuh")
KERNEL_SOURCES = {
    "volume": [os.path.join(_CSRC, f) for f in ("volume_kernel.cuh", "packed.cuh", "volume_inst.cu", "logmean_poly.inc") + _NUMERIC],
    "surface": [os.path.join(_CSRC, f) for f in ("surface_kernel.cu", "surface_index.cuh") + _NUMERIC],
}


def kernel_source_sha(kind: str = "volume") -> str:
    import hashlib
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kind]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_field(kernel: str, workload: str, field: str, kind: str = "volume"):
    """A field of a committed ncu summary's traffic_record, only if the kernel source is unchanged."""
    import glob
    sha = kernel_source_sha(kind)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_record:"):
                    rec = json.loads(line.split(":", 1)[1])
                    if rec["kernel"] == kernel and rec["workload"] == workload and rec["source_sha"] == sha:
                        return rec.get(field)
    return None


def recorded_traffic(kernel: str, workload: str, kind: str = "volume"):
    """DRAM bytes per launch (volume) or per three-launch call (surface) from a
    committed ncu summary, only if the kernel source is unchanged."""
    import glob
    sha = kernel_source_sha(kind)
    key = "dram_bytes_per_launch" if kind == "volume" else "dram_bytes_per_call"
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_record:"):
                    rec = json.loads(line.split(":", 1)[1])
                    if (rec["kernel"] == kernel and rec["workload"] == workload and rec["source_sha"] == sha
                            and key in rec):
                        return rec[key]
    return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        # samples "under load": the upper half by power draw
        if pw:
            cut = sorted(pw)[len(pw) // 2]
            loaded = [num(r[1]) for r in rows if num(r[3]) is not None and num(r[3]) >= cut and num(r[1])]
        else:
            loaded = sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
def element_shard(K: int, world: int, rank: int):
    """Contiguous, balanced element range (e_begin, e_count) of `rank` out of `world`.

    Elements are independent in the volume term, so ranks that each take one
    range need no exchange; the union of the ranges is 0..K exactly once."""
    base, extra = divmod(K, world)
    e_begin = rank * base + min(rank, extra)
    return e_begin, base + (1 if rank < extra else 0)


def rank_work(K: int, world: int, rank: int, split: bool):
    """Element range (e_begin, e_count) this rank evaluates: with --split, its
    element_shard range of the one mesh (strong scaling: the job's work is
    fixed and divided); otherwise the whole mesh (replicas: weak scaling)."""
    if split and world > 1:
        return element_shard(K, world, rank)
    return 0, K


def job_nodes(n: int, world: int, split: bool) -> int:
    """Nodes the whole job evaluates per step: one mesh when split, one per rank
    otherwise."""
    return n if (split and world > 1) else world * n


def max_over_ranks(x: float, group=None, device=None) -> float:
    """Largest value over all ranks (the timing rule: the slowest rank counts)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _setup(cfg, device):
    import torch

    import flux_differencing_gb300 as fd
    import workloads as wl

    g = wl.generate(cfg, device=device)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, cfg.precision, bc=cfg.bc)
    op.J = torch.empty(cfg.n, dtype=op.dtype, device=device)
    Ja = op.set_geometry(g["x"], g["y"], g["z"], J_out=op.J)
    q = g["q"].to(op.dtype).contiguous()
    phi = g["phi"].to(op.dtype).contiguous()
    del g
    out = torch.zeros((5, cfg.n), dtype=op.dtype, device=device)
    torch.cuda.synchronize(device)
    return op, q, Ja, phi, out


def _time_device(op, q, Ja, phi, out, steps, warmup, stream, barrier, what="volume", erange=None):
    """Per-call times with CUDA events on the launching stream.

    what: "volume" (one launch), "surface" (three launches, accumulating into
    out), "rhs" (esdg_rhs: four launches, one for FP32), "step" (one five-stage
    Runge-Kutta step: 5 to 25 launches, on a copy of q) or "stage" (one
    Runge-Kutta stage update)."""
    import torch

    if what in ("step", "stage"):
        qs = q.clone()
        dq = torch.zeros_like(q)
    # inputs made on the default stream must be complete before the timing stream reads them
    torch.cuda.synchronize()

    def call():
        if what == "volume":
            if erange is None:
                op.volume_rhs(q, Ja, phi, out=out, stream=stream)
            else:  # one element range of the mesh (esdg_volume_rhs_range)
                op.volume_rhs(q, Ja, phi, out=out, stream=stream, e_begin=erange[0], e_count=erange[1])
        elif what == "surface":
            op.surface_rhs(q, Ja, phi, out, stream=stream)
        elif what == "rhs":
            op.rhs(q, Ja, phi, out=out, stream=stream)
        elif what == "step":
            op.lsrk_step(qs, dq, out, Ja, phi, op.J, STEP_DT, stream=stream)
        else:  # one Runge-Kutta stage update (dt = 0 leaves the state unchanged)
            op.rk_stage(qs, dq, out, op.J, 0.5, 0.5, 0.0, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        barrier()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for k in range(steps):
            call()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    total = ev[0].elapsed_time(ev[steps])
    return total, per


def _time_e2e(op, q, Ja, phi, out, steps, warmup, stream, barrier):
    """Same metric through host buffers: pinned H2D of q, metrics, phi, the kernel, D2H of out."""
    import torch

    hq = q.cpu().pin_memory()
    hJ = Ja.cpu().pin_memory()
    hp = phi.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = (hq.numel() + hJ.numel() + hp.numel()) * hq.element_size()
    d2h = ho.numel() * ho.element_size()

    def step():
        q.copy_(hq, non_blocking=True)
        Ja.copy_(hJ, non_blocking=True)
        phi.copy_(hp, non_blocking=True)
        op.volume_rhs(q, Ja, phi, out=out, stream=stream)
        ho.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    return e0.elapsed_time(e1), h2d, d2h


E2E_WINDOWS = 3  # timed windows of the end-to-end loop; the median is reported


def _time_e2e_pipeline(op, q, Ja, phi, steps, warmup, barrier, depth=2, windows=E2E_WINDOWS):
    """The metric through the C-ABI's host-buffer pipeline (esdg_pipeline_*):
    every step submits the pinned host inputs (q, metrics, phi) and receives
    the result in a pinned host buffer; `depth` slots let one step's copies
    overlap another's kernel.  Host wall clock around the submissions, with
    the device synchronised on both sides (the slots' streams are the
    library's own).  `windows` timed windows of `steps` steps each; returns
    the median window's time (the host link is shared with other tenants of
    the machine, and a single window can catch their traffic), the bytes
    copied per step and the list of window times."""
    import time

    import torch

    import flux_differencing_gb300 as fd

    hq = q.cpu().pin_memory()
    hJ = Ja.cpu().pin_memory()
    hp = phi.cpu().pin_memory()
    houts = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(depth)]
    h2d = (hq.numel() + hJ.numel() + hp.numel()) * hq.element_size()
    d2h = houts[0].numel() * houts[0].element_size()
    pipe = fd.Pipeline(op, depth)
    times = []
    try:
        for k in range(warmup):
            pipe.submit(hq, hJ, hp, houts[k % depth])
        pipe.wait()
        torch.cuda.synchronize()
        for _ in range(windows):
            barrier()
            t0 = time.perf_counter()
            for k in range(steps):
                pipe.submit(hq, hJ, hp, houts[k % depth])
            pipe.wait()
            t1 = time.perf_counter()
            barrier()
            times.append((t1 - t0) * 1e3)
    finally:
        pipe.close()
    return statistics.median(times), h2d, d2h, times


def _fma_peak(fp64: bool, device) -> float:
    """Best-of-3 FMA throughput (FLOP/s) of the bench kernel over all SMs."""
    import ctypes

    import torch

    import flux_differencing_gb300 as fd
    lib = fd.load_library()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    blocks, threads = sms * 8, 256
    iters = 4096 if fp64 else 65536
    dt = torch.float64 if fp64 else torch.float32
    sink = torch.zeros(blocks, dtype=dt, device=device)
    s = torch.cuda.current_stream(device)
    best = 0.0
    for _ in range(4):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        rc = lib.esdg_bench_fma(1 if fp64 else 0, blocks, threads, iters, ctypes.c_void_p(sink.data_ptr()),
                                ctypes.c_void_p(s.cuda_stream))
        e1.record(s)
        torch.cuda.synchronize(device)
        if rc != 0:
            return float("nan")
        ms = e0.elapsed_time(e1)
        best = max(best, 16.0 * iters * blocks * threads / (ms * 1e-3))
    return best


def _cpu_baseline(cfg, budget_s: float = 12.0):
    """The oracle as it stands on this host's cores, on a bounded sample of elements."""
    import oracle
    import workloads as wl

    oracle.build()
    nthreads = oracle.max_threads()
    # pilot on a few elements to size the sample
    pilot = np.arange(min(cfg.K, max(8, nthreads)))
    g = wl.generate_elements(cfg, pilot)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, len(pilot), gc["x"], gc["y"], gc["z"])
    t0 = time.perf_counter()
    oracle.volume(cfg.N, len(pilot), gc["q"], Ja, gc["phi"], nthreads=nthreads)
    dt = max(time.perf_counter() - t0, 1e-4)
    count = int(min(cfg.K, max(len(pilot), len(pilot) * budget_s / dt)))
    elems = np.arange(count)
    g = wl.generate_elements(cfg, elems)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, count, gc["x"], gc["y"], gc["z"])
    t0 = time.perf_counter()
    oracle.volume(cfg.N, count, gc["q"], Ja, gc["phi"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    nodes = count * cfg.Nq ** 3
    single = _cpu_single_core(cfg, min(3.0, budget_s / 4))
    return {"value": nodes / dt / 1e9, "unit": "GDOF/s", "cores": nthreads, "kind": "oracle",
            "sample": f"first {count} of {cfg.K} elements of {cfg.name} ({nodes} nodes), FP64 oracle, "
                      f"{dt:.1f} s, OpenMP over elements",
            "elements": count, "single_core": single}


def _cpu_single_core(cfg, budget_s: float = 2.0):
    """The oracle on one host core (a bounded prefix of the workload's elements)."""
    import oracle
    import workloads as wl

    pilot = np.arange(min(cfg.K, 4))
    g = wl.generate_elements(cfg, pilot)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, len(pilot), gc["x"], gc["y"], gc["z"])
    t0 = time.perf_counter()
    oracle.volume(cfg.N, len(pilot), gc["q"], Ja, gc["phi"], nthreads=1)
    dt = max(time.perf_counter() - t0, 1e-4)
    count = int(min(cfg.K, max(len(pilot), len(pilot) * budget_s / dt)))
    g = wl.generate_elements(cfg, np.arange(count))
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, count, gc["x"], gc["y"], gc["z"])
    t0 = time.perf_counter()
    oracle.volume(cfg.N, count, gc["q"], Ja, gc["phi"], nthreads=1)
    dt = time.perf_counter() - t0
    nodes = count * cfg.Nq ** 3
    return {"value": nodes / dt / 1e9, "unit": "GDOF/s", "cores": 1,
            "sample": f"first {count} of {cfg.K} elements of {cfg.name}, {dt:.1f} s"}


PARITY_TOL = {"fp64": 1e-11, "fp32": 1e-4, "fp64ff": 1e-11}
VARS = ("rho", "rho_u1", "rho_u2", "rho_u3", "E")


def oracle_reference(cfg, elems, with_inputs=False):
    """The oracle's volume term and term scale S (per node and variable) on
    the given elements of a workload (FP64, OpenMP over elements); with_inputs
    also returns the elements' state, geopotential and oracle metrics."""
    import oracle
    import workloads as wl

    oracle.build()
    elems = np.asarray(elems)
    g = wl.generate_elements(cfg, elems)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, len(elems), gc["x"], gc["y"], gc["z"])
    out, scale = oracle.volume(cfg.N, len(elems), gc["q"], Ja, gc["phi"], with_scale=True,
                               nthreads=oracle.max_threads())
    if with_inputs:
        return out, scale, {"q": gc["q"], "phi": gc["phi"], "Ja": Ja}
    return out, scale


def kernel_only_parity(cfg, ref, scale, inputs, device):
    """The volume kernel on the sampled elements alone (a mesh of those
    elements), fed the oracle's own metric terms: its difference from the oracle
    is the kernel's arithmetic alone, without the rounding of the GPU's
    curl-form metrics that the end-to-end comparison also contains."""
    import torch

    import flux_differencing_gb300 as fd

    K = inputs["q"].shape[1] // cfg.Nq ** 3
    op = fd.VolumeOperator(K, 1, 1, cfg.N, cfg.precision)
    q = torch.from_numpy(np.ascontiguousarray(inputs["q"])).to(device, op.dtype)
    Ja = torch.from_numpy(np.ascontiguousarray(inputs["Ja"])).to(device, op.dtype)
    phi = torch.from_numpy(np.ascontiguousarray(inputs["phi"])).to(device, op.dtype)
    out = op.volume_rhs(q, Ja, phi)
    torch.cuda.synchronize(device)
    got = out.double().cpu().numpy()
    op.close()
    return parity_numbers(got, ref, scale, cfg.precision)


def parity_numbers(got, ref, scale, precision):
    """Per conserved variable: the normalised error e_c = max|gpu - oracle| / S_c
    (S_c = max_i sum |2 D (F + G)_c|, the magnitude of the terms the sum adds),
    the plain relative error max|gpu - oracle| / max|oracle| and the
    conditioning kappa_c = S_c / max|oracle_c| that separates the two."""
    rows = {}
    for c, name in enumerate(VARS):
        d = float(np.max(np.abs(got[c] - ref[c])))
        S = float(np.max(scale[c]))
        o = float(np.max(np.abs(ref[c])))
        rows[name] = {"e_c": d / S, "plain": d / o if o > 0 else None, "kappa": S / o if o > 0 else None}
    worst = max(r["e_c"] for r in rows.values())
    return {"max_e_c": worst, "tolerance": PARITY_TOL[precision], "pass": bool(worst <= PARITY_TOL[precision]),
            "per_variable": rows}


def _same_mesh(a, b):
    """Whether two workloads share mesh and state (the FP32 and float-float
    variants of a workload do; only the precision differs)."""
    return (a.N, a.Kx, a.Ky, a.Kz, a.state, a.domain, a.warp, a.seed) == (b.N, b.Kx, b.Ky, b.Kz, b.state,
                                                                          b.domain, b.warp, b.seed)


def gpu_rows(out_host, cfg, elems):
    """Columns of the given elements from a (5, n) host array of the whole mesh."""
    np3 = cfg.Nq ** 3
    idx = (np.asarray(elems)[:, None] * np3 + np.arange(np3)[None, :]).ravel()
    return out_host[:, idx]


ISSUE_PEAK_WARP_INST_PER_S = 152 * 4 * 2.07e9  # one warp instruction per SMSP and cycle at the top SM clock


def issue_roofline(kernel, cfg, t_s):
    """Instruction-issue roofline of a kernel that is bound by issue rather than
    by one pipe (float-float; packed FP32): warp instructions per launch from
    the committed ncu record of the same source (thread instructions per node
    / 32) over the launch time, against one issue per SMSP and cycle."""
    per_node = recorded_field(kernel, cfg.name, "inst_per_node")
    if per_node is None:
        return None
    rate = per_node / 32.0 * cfg.n / t_s
    return {"bound": "issue", "achieved": rate / 1e9, "peak": ISSUE_PEAK_WARP_INST_PER_S / 1e9,
            "unit": "G warp instructions/s", "frac": rate / ISSUE_PEAK_WARP_INST_PER_S,
            "inst_per_node": per_node,
            "source": "ncu instruction count of the committed profile (same kernel source); peak = 152 SMs x 4 "
                      "schedulers x 2.07 GHz"}


def run_oracle_sweep(args):
    """The oracle on the host: all cores and one core, on the three fixed configs
    (tiny box N = 3, bubble N = 4, channel N = 7); one JSON line each."""
    for name in ("tiny_box_N3", "bubble_N4", "channel_N7"):
        cfg = _wl().get_config(name)
        allc = _cpu_baseline(cfg, args.cpu_seconds)
        print(json.dumps({"sweep": "oracle", "config": name, "N": cfg.N, "nodes": cfg.n,
                          "all_cores_GDOF/s": allc["value"], "cores": allc["cores"],
                          "single_core_GDOF/s": allc["single_core"]["value"],
                          "samples": [allc["sample"], allc["single_core"]["sample"]]}), flush=True)


def _wl():
    import workloads as wl
    return wl


def run_reference(args):
    """--impl reference: the oracle timed on the host cores on the same workload."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    import workloads as wl

    cfg = wl.get_config(args.workload)
    oracle.build()
    nthreads = oracle.max_threads()
    per_step = max(1, min(cfg.K, args.ref_elements))
    elems = np.arange(per_step)
    g = wl.generate_elements(cfg, elems)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(cfg.N, per_step, gc["x"], gc["y"], gc["z"])
    for _ in range(args.warmup):
        oracle.volume(cfg.N, per_step, gc["q"], Ja, gc["phi"], nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.volume(cfg.N, per_step, gc["q"], Ja, gc["phi"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    nodes = per_step * cfg.Nq ** 3
    val = nodes * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": "volume-term GDOF/s (FP64)", "value": val, "unit": "GDOF/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg.name, "N": cfg.N, "K": cfg.K, "nodes": cfg.n,
                   "sample_elements_per_step": per_step},
        "cpu_baseline": {"value": val, "unit": "GDOF/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"first {per_step} elements of {cfg.name} per step"},
        "e2e": {"value": val, "unit": "GDOF/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import workloads as wl

    # each workload argument feeds the report section of its own precision
    for flag, wname, prec in (("--workload", args.workload, "fp64"), ("--fp32-workload", args.fp32_workload, "fp32"),
                              ("--ff-workload", args.ff_workload, "fp64ff")):
        if wname and wl.get_config(wname).precision != prec:
            raise SystemExit(f"{flag} {wname}: expected a {prec} workload")
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    def barrier():
        if ws > 1:
            dist.barrier()

    def slowest(x: float) -> float:
        return max_over_ranks(x, device=device)

    stream = torch.cuda.Stream(device)
    results = {}
    clocks = None
    # --split: the ranks divide one mesh by element ranges (no exchange: the
    # volume term is element-local); the surface term, the time step and the
    # host-buffer pipeline need the whole mesh (or a face halo) and are skipped
    split = bool(args.split and ws > 1)
    if split:
        args.no_surface = args.no_e2e = True
        args.large = ""
    extra = [w for w in (args.fp32_workload, args.ff_workload) if w]
    for wname in [args.workload] + extra:
        cfg = wl.get_config(wname)
        op, q, Ja, phi, out = _setup(cfg, device)
        sampler = ClockSampler(local) if (rank == 0 and wname == args.workload) else None
        if sampler:
            sampler.start()
        e_range = rank_work(cfg.K, ws, rank, args.split)
        total_ms, per = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier,
                                     erange=e_range if split else None)
        if sampler:
            clocks = sampler.stop()
        assert op.status() == 0, "non-physical state in the bench inputs"
        out_host = out.double().cpu().numpy() if (rank == 0 and not args.no_parity) else None
        total_ms = slowest(total_ms)
        ms = total_ms / args.steps
        gdof = job_nodes(cfg.n, ws, args.split) / (ms * 1e-3) / 1e9
        fl = flops_per_dof(cfg.N) * cfg.n
        res = {"cfg": cfg, "ms": ms, "gdof": gdof, "per": per,
               "flops_per_launch": fl, "achieved_tflops": fl / (statistics.mean(per) * 1e-3) / 1e12,
               "bytes_per_launch": BYTES_PER_DOF[cfg.precision] * cfg.n, "out_host": out_host}
        if not args.no_surface:
            s_total, s_per = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier,
                                          what="surface")
            r_total, r_per = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier,
                                          what="rhs")
            assert op.status() == 0, "non-physical state in the bench inputs"
            res["surface"] = {"ms": slowest(s_total) / args.steps, "per": s_per,
                              "rhs_ms": slowest(r_total) / args.steps}
            if not args.no_step:
                st_total, _ = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier,
                                           what="step")
                assert op.status() == 0, "non-physical state during the Runge-Kutta steps"
                k_total, k_per = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier,
                                              what="stage")
                assert op.status() == 0, "non-physical state during the Runge-Kutta stages"
                res["step"] = {"ms": slowest(st_total) / args.steps, "stage_ms": slowest(k_total) / args.steps,
                               "stage_per": k_per}
        if cfg.precision == "fp32" and not args.no_surface:
            # perturbation variables about the hydrostatic background (same kernels,
            # two more planes read, pressure formed from the perturbations)
            ref = wl.reference_state(cfg, device=device)
            rr = ref["rho_ref"].to(op.dtype).contiguous()
            pr = ref["p_ref"].to(op.dtype).contiguous()
            qp = q.clone()
            qp[0] = (q[0].double() - ref["rho_ref"]).to(op.dtype)
            qp[4] = (q[4].double() - (ref["p_ref"] / (GAMMA - 1.0) + ref["rho_ref"] * phi.double())).to(op.dtype)
            op.set_reference(rr, pr)
            torch.cuda.synchronize()
            pv_total, _ = _time_device(op, qp, Ja, phi, out, args.steps, args.warmup, stream, barrier)
            pr_total, _ = _time_device(op, qp, Ja, phi, out, args.steps, args.warmup, stream, barrier, what="rhs")
            assert op.status() == 0, "non-physical state in the perturbation inputs"
            op.set_reference()
            res["perturbation"] = {"volume_ms": slowest(pv_total) / args.steps,
                                   "rhs_ms": slowest(pr_total) / args.steps}
            del ref, rr, pr, qp
        if not args.no_e2e:
            e2e_steps = max(3, min(args.steps, 20))
            p_ms, h2d, d2h, p_windows = _time_e2e_pipeline(op, q, Ja, phi, e2e_steps, 6, barrier)
            p_ms = slowest(p_ms) / e2e_steps
            e_ms, _, _ = _time_e2e(op, q, Ja, phi, out, e2e_steps, 1, stream, barrier)
            e_ms = slowest(e_ms) / e2e_steps
            res["e2e"] = {"value": ws * cfg.n / (p_ms * 1e-3) / 1e9, "unit": "GDOF/s",
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": p_ms,
                          "api": "esdg_pipeline_submit (host buffers, two slots: one step's copies overlap "
                                 "another step's kernel)",
                          "timing": f"median of {E2E_WINDOWS} wall-clock windows of {e2e_steps} steps, each "
                                    "step with its copies in and out",
                          "window_ms_per_step": [round(w / e2e_steps, 4) for w in p_windows],
                          "serial": {"value": ws * cfg.n / (e_ms * 1e-3) / 1e9, "ms_per_step": e_ms,
                                     "how": "copy in, kernel, copy out on one stream, one step at a time"}}
        results[wname] = res
        op.close()
        del q, Ja, phi, out
        torch.cuda.empty_cache()

    # the largest single-GPU configuration (order sweep at N = 7, about 6.4e7
    # nodes), FP64 and FP32, each with its own clock record and a sampled parity
    large = []
    for wname in [w for w in (args.large or "").split(",") if w]:
        cfg = wl.get_config(wname)
        op, q, Ja, phi, out = _setup(cfg, device)
        sampler = ClockSampler(local) if rank == 0 else None
        if sampler:
            sampler.start()
        total_ms, per = _time_device(op, q, Ja, phi, out, args.steps, args.warmup, stream, barrier)
        lclocks = sampler.stop() if sampler else None
        assert op.status() == 0, "non-physical state in the bench inputs"
        ms = slowest(total_ms) / args.steps
        entry = {"cfg": cfg, "ms": ms, "per": per, "clocks": lclocks}
        if rank == 0 and not args.no_parity:
            elems = np.asarray(wl.element_subset(cfg, min(cfg.K, args.parity_sample)))
            np3 = cfg.Nq ** 3
            idx = torch.from_numpy((elems[:, None] * np3 + np.arange(np3)[None, :]).ravel()).to(device)
            entry["parity_elems"] = elems
            entry["gpu_rows"] = out[:, idx].double().cpu().numpy()
        large.append(entry)
        op.close()
        del q, Ja, phi, out
        torch.cuda.empty_cache()

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = _peaks()
    if args.no_peaks:
        fp64_meas, fp32_meas = float("nan"), float("nan")
    else:
        fp64_meas = _fma_peak(True, device) / 1e12
        fp32_meas = _fma_peak(False, device) / 1e12
    main = results[args.workload]
    cfg = main["cfg"]
    peak64 = max(NOMINAL_FP64_TFLOPS, fp64_meas) if fp64_meas == fp64_meas else NOMINAL_FP64_TFLOPS
    traffic = recorded_traffic(f"volume_kernel<double, {cfg.N}>", cfg.name)
    roof = {"bound": "alu", "achieved": main["achieved_tflops"], "peak": peak64, "unit": "TFLOP/s",
            "frac": main["achieved_tflops"] / peak64, "traffic": traffic,
            "traffic_unit": "bytes per launch (ncu dram read + write)",
            "peak_source": f"FP64 vector FMA: max(nominal {NOMINAL_FP64_TFLOPS}, measured {fp64_meas:.3f}) TFLOP/s",
            "algorithmic_flops_per_dof": flops_per_dof(cfg.N),
            "hardware": _hw_flops(cfg, main, peak64),
            "hbm": {"achieved_gbs": main["bytes_per_launch"] / (statistics.mean(main["per"]) * 1e-3) / 1e9,
                    "peak_gbs": peaks.get("hbm_gbs"), "peak_source": peak_src}}
    line = {
        "metric": "volume-term GDOF/s (FP64)", "value": main["gdof"], "unit": "GDOF/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms"], "higher_is_better": True,
        "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "N": cfg.N, "K": cfg.K, "elements": [cfg.Kx, cfg.Ky, cfg.Kz],
                   "nodes": cfg.n, "precision": cfg.precision, "form": "2d",
                   "l2": f"inputs {15 * cfg.n * 8 / 1e6:.0f} MB > 129 MB L2, no flush",
                   "parallelism": (f"one mesh split into {ws} contiguous element ranges (esdg_volume_rhs_range), "
                                   "no exchange" if split else f"elements, {ws} rank(s) with a mesh each, "
                                   "no exchange")},
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if "e2e" in main:
        line["e2e"] = {k: v for k, v in main["e2e"].items() if k != "ms_per_step"}
        line["gpu_launches"] += (E2E_WINDOWS + 1) * max(3, min(args.steps, 20))  # pipelined and serial end-to-end loops
    if args.fp32_workload:
        r32 = results[args.fp32_workload]
        c32 = r32["cfg"]
        hbm32 = r32["bytes_per_launch"] / (statistics.mean(r32["per"]) * 1e-3) / 1e9
        line["fp32"] = {
            "workload": c32.name, "value": r32["gdof"], "unit": "GDOF/s", "ms_per_step": r32["ms"],
            "roofline": {"bound": "alu", "achieved": r32["achieved_tflops"], "peak": fp32_meas,
                         "unit": "TFLOP/s", "frac": r32["achieved_tflops"] / fp32_meas,
                         "traffic": recorded_traffic(f"volume_kernel<float, {c32.N}>", c32.name),
                         "peak_source": "measured FP32 vector FMA",
                         "hbm": {"achieved_gbs": hbm32, "peak_gbs": peaks.get("hbm_gbs"),
                                 "frac": hbm32 / peaks["hbm_gbs"] if peaks.get("hbm_gbs") else None},
                         "issue": issue_roofline(f"volume_kernel<float, {c32.N}>", c32,
                                                 statistics.mean(r32["per"]) * 1e-3)},
        }
        if "e2e" in r32:
            line["fp32"]["e2e"] = {k: v for k, v in r32["e2e"].items() if k != "ms_per_step"}
        if "perturbation" in r32:
            pt = r32["perturbation"]
            line["fp32"]["perturbation"] = {
                "what": "perturbation variables about the hydrostatic background (esdg_set_reference)",
                "volume_ms": pt["volume_ms"], "volume_GDOF/s": ws * c32.n / (pt["volume_ms"] * 1e-3) / 1e9,
                "rhs_ms": pt["rhs_ms"], "overhead_vs_full_state": pt["volume_ms"] / r32["ms"] - 1.0}
            line["gpu_launches"] += (1 + rhs_launches("fp32")) * args.steps  # volume and rhs timings
        line["gpu_launches"] += args.steps + ((E2E_WINDOWS + 1) * max(3, min(args.steps, 20)) if "e2e" in r32 else 0)
    if args.ff_workload:
        rf = results[args.ff_workload]
        cf = rf["cfg"]
        # FP64 results from float-float pair arithmetic on the FP32 pipes: the
        # roofline is the FP32 vector peak (the FP64 pipe only converts and
        # computes the per-node logarithms)
        line["fp64ff"] = {
            "workload": cf.name, "value": rf["gdof"], "unit": "GDOF/s", "ms_per_step": rf["ms"],
            "dtype": "f64 storage, f32x2 (float-float) arithmetic",
            "speedup_vs_fp64": main["ms"] / rf["ms"],
            # the float-float arithmetic runs on the FP32 pipes and is bound by
            # instruction issue, not by one pipe: its roofline is the issue rate
            "roofline": issue_roofline(f"volume_kernel<double, {cf.N}, ff>", cf, statistics.mean(rf["per"]) * 1e-3),
            "algorithmic_fp64_equivalent_TFLOP/s": rf["achieved_tflops"],
            "traffic": recorded_traffic(f"volume_kernel<double, {cf.N}, ff>", cf.name),
        }
        if "e2e" in rf:
            line["fp64ff"]["e2e"] = {k: v for k, v in rf["e2e"].items() if k != "ms_per_step"}
        line["gpu_launches"] += args.steps + ((E2E_WINDOWS + 1) * max(3, min(args.steps, 20)) if "e2e" in rf else 0)
    if "surface" in main:
        line["surface"] = _surface_report(cfg, main["surface"], ws, peak64, "FP64 vector", peaks.get("hbm_gbs"))
        line["gpu_launches"] += (3 + rhs_launches(cfg.precision)) * args.steps  # surface and rhs timings
    for key, wname in (("main", args.workload), ("fp32", args.fp32_workload), ("fp64ff", args.ff_workload)):
        if wname and "step" in results[wname]:
            rep = _step_report(results[wname]["cfg"], results[wname], ws, peaks.get("hbm_gbs"))
            (line if key == "main" else line[key])["step"] = rep
            # the step's launches plus the standalone stage timing (one per step)
            line["gpu_launches"] += (rep["launches_per_step"] + 1) * args.steps
    if args.fp32_workload and "surface" in results[args.fp32_workload]:
        r32 = results[args.fp32_workload]
        line["fp32"]["surface"] = _surface_report(r32["cfg"], r32["surface"], ws, fp32_meas, "FP32 vector",
                                                  peaks.get("hbm_gbs"))
        line["gpu_launches"] += (3 + rhs_launches("fp32")) * args.steps
    if args.ff_workload and "surface" in results[args.ff_workload]:
        rf = results[args.ff_workload]
        line["fp64ff"]["surface"] = _surface_report(rf["cfg"], rf["surface"], ws, None,
                                                    "none: float-float on the FP32 pipes, latency-bound",
                                                    peaks.get("hbm_gbs"))
        line["gpu_launches"] += (3 + rhs_launches("fp64ff")) * args.steps
    line["peaks_measured"] = {"fp64_tflops": fp64_meas, "fp32_tflops": fp32_meas}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(cfg, args.cpu_seconds)
    if not args.no_parity:
        # every timed kernel's output against the oracle, element by element, on
        # the elements the CPU baseline covered (the whole mesh when it fits)
        count = line.get("cpu_baseline", {}).get("elements") or min(cfg.K, args.parity_sample)
        count = min(count, rank_work(cfg.K, ws, 0, split)[1])  # rank 0 holds its own range only
        elems = np.arange(count)
        ref, scale, inputs = oracle_reference(cfg, elems, with_inputs=True)
        par = {"sample": f"first {count} of {cfg.K} elements of {cfg.name}",
               "oracle": "FP64 oracle on the FP64 inputs (FP32 kernel: its inputs are those rounded to FP32)",
               "kernel_only": "the same kernel on the sampled elements fed the oracle's own metric terms "
                              "(the kernel's arithmetic alone; the main figures also contain the rounding "
                              "of the GPU's curl-form metrics)"}
        for key, wname in (("fp64", args.workload), ("fp32", args.fp32_workload), ("fp64ff", args.ff_workload)):
            if wname and results[wname].get("out_host") is not None and \
                    (wname == args.workload or _same_mesh(results[wname]["cfg"], cfg)):
                wc = results[wname]["cfg"]
                par[key] = parity_numbers(gpu_rows(results[wname]["out_host"], cfg, elems), ref, scale,
                                          wc.precision)
                par[key]["kernel_only"] = kernel_only_parity(wc, ref, scale, inputs, device)["per_variable"]
        line["parity"] = par
    if large:
        line["largest"] = []
        for ent in large:
            lc = ent["cfg"]
            t = statistics.mean(ent["per"]) * 1e-3
            fl = flops_per_dof(lc.N) * lc.n
            ach = fl / t / 1e12
            pk = peak64 if lc.precision == "fp64" else fp32_meas
            hbm = BYTES_PER_DOF[lc.precision] * lc.n / t / 1e9
            rep = {"workload": lc.name, "precision": lc.precision, "N": lc.N,
                   "elements": [lc.Kx, lc.Ky, lc.Kz], "nodes": lc.n,
                   "value": ws * lc.n / (ent["ms"] * 1e-3) / 1e9, "unit": "GDOF/s", "ms_per_step": ent["ms"],
                   "roofline": {"bound": "alu", "achieved": ach, "peak": pk, "unit": "TFLOP/s",
                                "frac": ach / pk if pk == pk else None,
                                "peak_source": ("FP64" if lc.precision == "fp64" else "FP32") + " vector FMA",
                                "hbm": {"achieved_gbs": hbm, "peak_gbs": peaks.get("hbm_gbs"),
                                        "frac": hbm / peaks["hbm_gbs"] if peaks.get("hbm_gbs") else None}},
                   "clocks": ent["clocks"]}
            if "gpu_rows" in ent:
                r2, sc2, inp2 = oracle_reference(lc, ent["parity_elems"], with_inputs=True)
                rep["parity"] = dict(parity_numbers(ent["gpu_rows"], r2, sc2, lc.precision),
                                     sample=f"{len(ent['parity_elems'])} elements spread over the mesh "
                                            f"(first and last included)")
                rep["parity"]["kernel_only"] = kernel_only_parity(lc, r2, sc2, inp2, device)["per_variable"]
            line["largest"].append(rep)
            line["gpu_launches"] += args.steps
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _hw_flops(cfg, res, peak_tflops):
    """FP64 FLOP/s counted by the hardware (dadd + dmul + 2 dfma per node from the
    committed ncu summary of this kernel and workload) over the bench's own
    launch time: the measure a "% of FP64 peak" target refers to.  Null when
    the kernel source changed since the capture."""
    per_node = recorded_field(f"volume_kernel<double, {cfg.N}>", cfg.name, "fp64_hw_flops_per_node")
    if per_node is None:
        return None
    t = statistics.mean(res["per"]) * 1e-3
    ach = per_node * cfg.n / t / 1e12
    return {"flops_per_node": per_node, "achieved_tflops": ach, "frac": ach / peak_tflops,
            "source": "ncu instruction counts of the committed volume profile (same kernel source)"}


def _surface_report(cfg, sres, ws, alu_peak_tflops, alu_peak_name, hbm_peak_gbs):
    """Surface-term and volume+surface lines for one workload (three direction
    launches per surface call, accumulated into the volume output)."""
    inner, walls = surface_counts(cfg)
    es = 4 if cfg.precision == "fp32" else 8
    flops = SURF_IFACE_OPS * inner + SURF_WALL_OPS * walls
    nbytes = es * (SURF_IFACE_VALUES * inner + SURF_WALL_VALUES * walls)
    t = statistics.mean(sres["per"]) * 1e-3
    tfl = flops / t / 1e12
    gbs = nbytes / t / 1e9
    f_alu = tfl / alu_peak_tflops if (alu_peak_tflops is not None and alu_peak_tflops == alu_peak_tflops) else None
    f_hbm = gbs / hbm_peak_gbs if hbm_peak_gbs else None
    bound = "hbm" if (f_hbm or 0) >= (f_alu or 0) else "alu"
    kname = {"fp64": "surface_kernel<double>", "fp32": "surface_kernel<float>",
             "fp64ff": "surface_kernel<double, ff>"}[cfg.precision]
    traffic = recorded_traffic(kname, cfg.name, kind="surface")
    return {
        "workload": cfg.name, "bc": list(cfg.bc),
        "surface": {"ms_per_call": sres["ms"], "launches_per_call": 3,
                    "GDOF/s": ws * cfg.n / (sres["ms"] * 1e-3) / 1e9,
                    "face_nodes": {"interior": inner, "wall": walls},
                    "roofline": {"bound": bound,
                                 "achieved_GB/s": gbs, "hbm_peak_GB/s": hbm_peak_gbs, "hbm_frac": f_hbm,
                                 "achieved_TFLOP/s": tfl, "alu_peak_TFLOP/s": alu_peak_tflops,
                                 "alu_peak": alu_peak_name, "alu_frac": f_alu,
                                 "algorithmic_bytes_per_call": nbytes, "algorithmic_flops_per_call": flops,
                                 "traffic": traffic,
                                 "traffic_unit": "bytes per call (ncu dram read + write, three launches)"}},
        "rhs": {"what": "volume + surface (esdg_rhs)" + (": one launch, the volume kernel evaluating each "
                                                         "element's faces" if cfg.precision == "fp32" else ""),
                "ms_per_step": sres["rhs_ms"], "launches_per_step": rhs_launches(cfg.precision),
                "GDOF/s": ws * cfg.n / (sres["rhs_ms"] * 1e-3) / 1e9},
    }


def rhs_launches(precision: str) -> int:
    """Kernel launches of one esdg_rhs."""
    return 1 if precision == "fp32" else 4


def step_launches(precision: str) -> int:
    """Kernel launches of one esdg_lsrk_step (five stages)."""
    return {"fp64": 25, "fp64ff": 20, "fp32": 5}[precision]


_STEP_WHAT = {
    "fp64": "volume + surface (esdg_rhs), then the stage kernel",
    "fp64ff": "the surface term, then the volume kernel adding it and applying the stage update in its store",
    "fp32": "one launch: the volume kernel also evaluates its elements' faces (reading the neighbours' face "
            "traces) and applies the stage update in its store, q and rhs alternating as state buffers; "
            "one device copy of the state back to q per step",
}


def _step_report(cfg, res, ws, hbm_peak_gbs):
    """One five-stage Runge-Kutta step: time, throughput and per-kernel shares."""
    st = res["step"]
    es = 4 if cfg.precision == "fp32" else 8
    stage_t = statistics.mean(st["stage_per"]) * 1e-3
    gbs = RK_STAGE_VALUES * es * cfg.n / stage_t / 1e9
    srf = 5 * res["surface"]["ms"]
    if cfg.precision == "fp64":
        shares = {"volume": 5 * res["ms"] / st["ms"], "surface": srf / st["ms"],
                  "rk_stage": 5 * st["stage_ms"] / st["ms"]}
    elif cfg.precision == "fp64ff":
        shares = {"surface": srf / st["ms"], "volume_with_fused_update": 1.0 - srf / st["ms"]}
    else:
        # one fused launch per stage: its time over the plain volume kernel's
        shares = {"fused_stage_ms": st["ms"] / 5, "volume_only_ms": res["ms"],
                  "fused_over_volume_only": st["ms"] / 5 / res["ms"]}
    return {"what": "five-stage low-storage Runge-Kutta step (esdg_lsrk_step): per stage " + _STEP_WHAT[cfg.precision],
            "ms_per_step": st["ms"], "launches_per_step": step_launches(cfg.precision),
            "GDOF/s": ws * cfg.n / (st["ms"] * 1e-3) / 1e9,
            "shares": shares,
            "standalone_rk_stage": {"ms": st["stage_ms"], "bound": "hbm", "achieved_GB/s": gbs,
                                    "peak_GB/s": hbm_peak_gbs, "frac": gbs / hbm_peak_gbs if hbm_peak_gbs else None,
                                    "algorithmic_bytes_per_node": RK_STAGE_VALUES * es,
                                    "note": "esdg_rk_stage on its own; the step fuses this update into the "
                                            "volume kernel"}}


def run_graph_sweep(args, device, stream):
    """One five-stage time step of small meshes, launched eagerly (5-25
    launches per step from the host) and replayed from a CUDA graph captured
    once: where the kernels are short, the launch path is the cost."""
    import torch

    import workloads as wl

    cases = [wl.get_config("tiny_box_N3")]
    for N, k in ((3, 8), (7, 4), (7, 8)):
        for prec in ("fp64", "fp32"):
            cases.append(wl.small_config(N, K=(k, k, k), warp=True, precision=prec))
    steps = max(args.steps, 50)
    for cfg in cases:
        op, q, Ja, phi, out = _setup(cfg, device)
        dq = torch.zeros_like(q)
        qs = q.clone()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                op.lsrk_step(qs, dq, out, Ja, phi, op.J, STEP_DT, stream=stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                op.lsrk_step(qs, dq, out, Ja, phi, op.J, STEP_DT, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
        eager = e0.elapsed_time(e1) / steps
        graph = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream(device)
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                op.lsrk_step(qs, dq, out, Ja, phi, op.J, STEP_DT, stream=gs)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize()
        replay = g0.elapsed_time(g1) / steps
        assert op.status() == 0
        print(json.dumps({"sweep": "graph", "config": cfg.name, "N": cfg.N, "K": cfg.K, "nodes": cfg.n,
                          "precision": cfg.precision, "launches_per_step": step_launches(cfg.precision),
                          "eager_ms_per_step": eager, "graph_ms_per_step": replay,
                          "speedup": eager / replay}), flush=True)
        op.close()
        del q, Ja, phi, out, dq, qs
        torch.cuda.empty_cache()


def run_sweep(args):
    """Opt-in measurement sweeps, one JSON line per point on stdout.

    orders:   the ~6.4e7-node warped cube for N = 2..8 in FP64 and FP32
              (the order-sweep workloads).
    parity:   the named workloads (tiny box, bubble, channel, order sweep at
              N = 7) in each precision against the oracle: normalised error,
              plain relative error and conditioning per variable (whole mesh
              up to 4.2e6 nodes, a spread sample of elements beyond).
    Every point carries the SM clocks sampled during its timed region.
    elements: throughput against element count for several orders on a
              warped cube with K = k^3 elements (as in the paper's Fig. 5:
              single-GPU saturation), reported in GDOF/s and in thousands of
              element evaluations per second."""
    import torch

    import workloads as wl

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    points = []
    if args.sweep == "graph":
        run_graph_sweep(args, device, stream)
        return
    precs = [x for x in ("fp64", "fp32", "fp64ff") if x in args.precisions.split(",")]
    if args.sweep == "orders":
        for N in [int(v) for v in args.orders.split(",")]:
            for prec in precs:
                points.append(wl.get_config(f"sweep_N{N}" + {"fp64": "", "fp32": "_fp32", "fp64ff": "_ff"}[prec]))
    elif args.sweep == "parity":
        # the five named workloads in every precision (the FP32 and float-float
        # variants share mesh and state), compared with the oracle
        import dataclasses
        for name in ("tiny_box_N3", "bubble_N4", "channel_N7", "sweep_N7"):
            base = wl.get_config(name)
            for prec in precs:
                points.append(dataclasses.replace(base, name=f"{name}:{prec}", precision=prec))
    else:
        for N in (2, 4, 7, 8):
            for k in (2, 4, 8, 16, 32, 48, 64):
                if k ** 3 * (N + 1) ** 3 > 1.1e8:
                    continue
                for prec in precs:
                    points.append(wl.small_config(N, K=(k, k, k), warp=True, precision=prec))
    for cfg in points:
        op, q, Ja, phi, out = _setup(cfg, device)
        # short launches need more of them for a stable mean, and a timed
        # region long enough for the clock samples (100 ms apart)
        steps = max(args.steps, 3)
        _time_device(op, q, Ja, phi, out, 2, 1, stream, lambda: None)
        probe = (lambda t: t[0] / 2)(_time_device(op, q, Ja, phi, out, 2, 0, stream, lambda: None))
        steps = max(steps, int(0.5 / max(probe * 1e-3, 1e-6)))
        sampler = ClockSampler(0)
        sampler.start()
        total_ms, per = _time_device(op, q, Ja, phi, out, steps, args.warmup, stream, lambda: None)
        clocks = sampler.stop()
        ms = total_ms / steps
        line = {"sweep": args.sweep, "config": cfg.name, "N": cfg.N, "K": cfg.K, "nodes": cfg.n,
                "precision": cfg.precision, "ms_per_launch": ms, "GDOF/s": cfg.n / (ms * 1e-3) / 1e9,
                "kilo_element_evals_per_s": cfg.K / (ms * 1e-3) / 1e3,
                "algorithmic_TFLOP/s": flops_per_dof(cfg.N) * cfg.n / (ms * 1e-3) / 1e12,
                "HBM_GB/s": BYTES_PER_DOF[cfg.precision] * cfg.n / (ms * 1e-3) / 1e9,
                "steps": steps, "clocks": clocks}
        if args.sweep == "parity":
            elems = (np.arange(cfg.K) if cfg.n <= 1 << 22 else
                     np.asarray(wl.element_subset(cfg, min(cfg.K, args.parity_sample))))
            ref, scale, inputs = oracle_reference(cfg, elems, with_inputs=True)
            line["parity"] = dict(parity_numbers(gpu_rows(out.double().cpu().numpy(), cfg, elems), ref, scale,
                                                 cfg.precision),
                                  sample=f"{len(elems)} of {cfg.K} elements")
            line["parity"]["kernel_only"] = kernel_only_parity(cfg, ref, scale, inputs, device)["per_variable"]
        print(json.dumps(line), flush=True)
        op.close()
        del q, Ja, phi, out
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="channel_N7")
    ap.add_argument("--fp32-workload", default="channel_N7_fp32")
    ap.add_argument("--ff-workload", default="channel_N7_ff",
                    help="FP64 buffers with float-float pair arithmetic, reported under \"fp64ff\"")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-surface", action="store_true", help="skip the surface-term and full-RHS timings")
    ap.add_argument("--no-step", action="store_true", help="skip the Runge-Kutta step timing")
    ap.add_argument("--no-peaks", action="store_true", help="skip the FMA-throughput peak measurement")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-elements", type=int, default=256)
    ap.add_argument("--sweep", choices=["orders", "elements", "graph", "oracle", "parity"], default=None,
                    help="opt-in measurement sweeps (one JSON line per point) instead of the bench line")
    ap.add_argument("--precisions", default="fp64,fp32,fp64ff",
                    help="comma-separated precisions of the orders and elements sweeps")
    ap.add_argument("--orders", default="2,3,4,5,6,7,8", help="comma-separated orders N of the orders sweep")
    ap.add_argument("--large", default="sweep_N7,sweep_N7_fp32",
                    help="largest single-GPU workloads timed in the same run (comma-separated; '' for none)")
    ap.add_argument("--no-parity", action="store_true", help="skip the parity report against the oracle")
    ap.add_argument("--split", action="store_true",
                    help="under torchrun: divide one mesh among the ranks by element ranges (strong scaling) "
                         "instead of one mesh per rank (weak scaling)")
    ap.add_argument("--parity-sample", type=int, default=512,
                    help="elements compared with the oracle when the CPU baseline does not set the sample")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.fp32_workload in ("", "none"):
        args.fp32_workload = None
    if args.ff_workload in ("", "none"):
        args.ff_workload = None
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep == "oracle":
        run_oracle_sweep(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
