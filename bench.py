#!/usr/bin/env python
"""Throughput of the D3Q19 BGK stream-collide step on GB300, in MLUPS (million lattice-cell
updates per second, counting every cell), with the HBM roofline of the dominant kernel.

Workload (the headline): a 512^3 periodic porous medium (3x3x3 solid blobs until 30 % of the cells
are solid, seed 1005), body acceleration g = (1e-6, 0, 0) with Guo forcing, tau = 0.7, fluid at
rest, AA in-place streaming, stream (SoA) layout.  One benchmark step = lbm_step(ctx, 2): an even
and an odd AA step (the pattern's period), the second with the momentum-exchange force.
The population buffer (10.2 GB) is far larger than L2, so no L2 flush is needed between steps.

Also printed in the same JSON line: AA vs A-B at 128^3 and 512^3 on periodic boxes without solids
("variants"), an end-to-end figure through host buffers ("e2e"), the CPU oracle timed on a
bounded sample ("cpu_baseline"), SM clocks sampled during the timed region ("clocks").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl  # noqa: E402

METRIC = "MLUPS (D3Q19 fp32, AA vs A-B) at 128^3 and 512^3; % of HBM roofline"
UNIT = "MLUPS"
# population bytes per cell update ("GPU lattice Boltzmann: streaming layout and performance":
# 152 in place; the fused pull moves the same 19 reads + 19 writes) plus the 1-byte cell flag
POP_BYTES = 152
FLAG_BYTES = 1
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---- roofline helpers (host logic; tested on the CPU) ------------------------------------------------

def algorithmic_bytes(n_cells: int, scheme: str = "AA") -> float:
    """Bytes per launch of a step kernel by the bytes-per-update convention: 19 fp32 reads + 19
    writes and one flag byte per cell update, counting every cell (in a porous medium the 32-byte
    sectors of the population planes are moved for solid cells too; the measured DRAM traffic
    per cell agrees).  The two-pass A-B form moves twice the populations."""
    per_cell = (2 * POP_BYTES if scheme == "AB2" else POP_BYTES) + FLAG_BYTES
    return float(n_cells) * per_cell


def fluid_bytes(n_cells: int, n_fluid: int) -> float:
    """The populations the method itself needs: 152 B per FLUID cell, plus the flag bytes."""
    return float(n_fluid) * POP_BYTES + float(n_cells) * FLAG_BYTES


def roofline_glups(bandwidth_gbs: float, bytes_per_update: float) -> float:
    """Code-balance bound (PortLBM §5.2): updates per second = bandwidth / bytes per update."""
    return bandwidth_gbs / bytes_per_update


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_tokens(text: str) -> str:
    """C / C++ / CUDA source without its comments, runs of white space reduced to one blank:
    what the compiler sees, so that edits to comments leave it unchanged.  String and character
    literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """sha256 over the kernel sources' code (comments and layout of white space excluded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lattice_boltzmann_cfd_d3q19_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()


def recorded_traffic(kernel: str):
    """DRAM bytes per cell of `kernel` from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line and ":" in line:
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    v = rec.get(f"{kernel}_dram_bytes_per_cell")
    return float(v) if v else None


# ---- clocks --------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.out = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.out.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---- distributed plumbing (one process per GPU, independent replicas) ---------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of `value` over ranks (the slowest replica sets the whole-job time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_mlups(cells_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Units all ranks processed divided by the slowest rank's time (weak scaling)."""
    return world * cells_per_step * steps / max_seconds / 1e6


def workload_config(n, tau, g, fluid_fraction):
    """The `config` object of both arms: the porous workload and how it is timed."""
    N = n ** 3
    return {"workload": f"porous medium {n}^3, 30% solid in 3^3 blobs (seed 1005), periodic, "
                        "Guo body force gx=1e-6, tau=0.7, AA in place, stream (SoA) layout",
            "nx": n, "ny": n, "nz": n, "streaming": "AA", "layout": "stream",
            "tau": tau, "g": list(g), "fluid_fraction": round(fluid_fraction, 4),
            "lbm_steps_per_step": 2,
            "l2": (f"inputs larger than L2 ({19 * 4 * N / 1e9:.1f} GB population buffer vs "
                   "126 MB L2), no flush")}


# ---- the GPU arm ---------------------------------------------------------------------------------------

_POROUS_FLAGS = {}


def porous_flags(n):
    """The benchmark's porous medium at edge n (generated once per run)."""
    if n not in _POROUS_FLAGS:
        _POROUS_FLAGS[n] = wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512)
    return _POROUS_FLAGS[n]


def make_porous_context(B, torch, n, tau, g, scheme="AA"):
    flags = porous_flags(n)
    ctx = B.lbm_create(n, n, n, tau, B.LAYOUT_STREAM,
                       B.STREAMING_AA if scheme == "AA" else B.STREAMING_AB)
    B.lbm_set_flags(ctx, flags)
    B.lbm_set_body_force(ctx, *g)
    N = n ** 3
    rho = torch.ones(N, dtype=torch.float32, device="cuda")
    u = torch.zeros(3 * N, dtype=torch.float32, device="cuda")
    B.lbm_set_equilibrium(ctx, rho, u)
    return ctx, flags


def timed_steps(B, torch, ctx, steps, warmup, per_step=2, profile=True, sampler=None,
                world=1):
    stream = torch.cuda.current_stream()
    B.lbm_set_stream(ctx, stream.cuda_stream)
    for _ in range(warmup):
        B.lbm_step(ctx, per_step)
    torch.cuda.synchronize()
    if profile:
        B.lbm_profile_enable(ctx, True)
    if sampler:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = B.lbm_kernel_launches(ctx)
    # one event between consecutive steps: the region's time and each step's
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    e0, e1 = ev[0], ev[-1]
    e0.record(stream)
    for i in range(steps):
        B.lbm_step(ctx, per_step)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    launches = B.lbm_kernel_launches(ctx) - launches0
    prof = {}
    if profile:
        for kind, name in ((B.K_AA_EVEN, "aa_even"), (B.K_AA_ODD, "aa_odd"),
                           (B.K_AB_PULL, "ab_pull"), (B.K_AB_COLLIDE, "ab_collide"),
                           (B.K_BOUNDARY, "boundary"), (B.K_PREGATHER, "pregather"),
                           (B.K_FORCE, "force_reduce")):
            cnt, tot = B.lbm_profile_read(ctx, kind)
            if cnt:
                prof[name] = (cnt, tot)
        B.lbm_profile_enable(ctx, False)
    return ms, launches, prof, clocks, step_ms


def variant(B, torch, n, scheme, steps=10, warmup=3, cavity=False, fp16=False, layout="stream",
            sphere=False, porous=False):
    """Periodic box without solids, g = 0, uniform flow: the clean roofline point.  With
    cavity=True: a lid-driven cavity (resting walls, lid moving at 0.05 along x), fluid at rest.
    With sphere=True: the sphere workload (r = n/8 at (0.3125 n, n/2, n/2), equilibrium inlet
    u = (0.05, 0, 0) on x = 0, zero-gradient outlet, y/z periodic, tau 0.56, fluid at the inlet
    state).  With fp16=True the populations are stored in half precision (76 population bytes per
    update instead of 152; the roofline fraction uses those bytes).  `layout`: stream, bundle or
    collision (fp32).  With porous=True: the benchmark's porous medium (g = (1e-6, 0, 0), tau 0.7,
    fluid at rest)."""
    lay = {"stream": B.LAYOUT_STREAM, "bundle": B.LAYOUT_BUNDLE,
           "collision": B.LAYOUT_COLLISION}[layout]
    tau = 0.56 if sphere else 0.7 if porous else 0.6
    ctx = B.lbm_create(n, n, n, tau, B.LAYOUT_STREAM_FP16 if fp16 else lay,
                       B.STREAMING_AA if scheme == "AA" else B.STREAMING_AB)
    try:
        N = n ** 3
        if cavity:
            B.lbm_set_flags(ctx, wl.cavity_flags(n, n, n))
            B.lbm_set_wall_velocity(ctx, 0.05, 0.0, 0.0)
        if porous:
            B.lbm_set_flags(ctx, porous_flags(n))
            B.lbm_set_body_force(ctx, 1e-6, 0.0, 0.0)
        if sphere:
            B.lbm_set_flags(ctx, wl.sphere_flags(n, n, n, (5 * n // 16, n // 2, n // 2), n / 8))
            B.lbm_set_faces(ctx, B.OPEN, B.PERIODIC, B.PERIODIC)
            B.lbm_set_inlet(ctx, 1.0, 0.05, 0.0, 0.0)
        rho = torch.ones(N, dtype=torch.float32, device="cuda")
        u = torch.zeros(3 * N, dtype=torch.float32, device="cuda")
        if sphere:
            u[:N] = 0.05
        elif not cavity and not porous:
            u[:N] = 0.02
        B.lbm_set_equilibrium(ctx, rho, u)
        # throughput with graph replay (no per-kernel events), then per-kernel event timing
        ms, _, _, _, _ = timed_steps(B, torch, ctx, steps, warmup, profile=False)
        _, _, prof, _, _ = timed_steps(B, torch, ctx, steps, warmup)
    finally:
        B.lbm_destroy(ctx)
    mlups = N * 2 * steps / (ms / 1e3) / 1e6
    peak, _ = measured_peaks()
    per_cell = (POP_BYTES // 2 if fp16 else POP_BYTES) + FLAG_BYTES
    kernels = {}
    for name, (cnt, tot) in prof.items():
        if name == "force_reduce":
            continue
        if name in ("boundary", "pregather"):
            # small kernels over the special cells / open faces: time only
            kernels[name] = {"ms": round(tot / cnt, 4)}
            continue
        gbs = N * per_cell / (tot / cnt / 1e3) / 1e9
        kernels[name] = {"ms": round(tot / cnt, 4), "GB/s": round(gbs, 1),
                         "frac": round(gbs / peak, 4)}
    return {"mlups": round(mlups, 1), "ms_per_lbm_step": round(ms / (2 * steps), 4),
            "bytes_per_update": per_cell,
            "frac_of_roofline": round(mlups * 1e6 * per_cell / 1e9 / peak, 4),
            "kernels": kernels}


def slab_variant(B, torch, n, world, steps=10, warmup=3):
    """The porous n^3 medium (A-B scheme) as `world` z slabs of one context each, all on this GPU:
    each slab holds its owned planes and two ghost planes, and the host moves the halo buffers
    between the slabs with device copies.  Timed three ways, one LBM step per step: the unsliced
    context (lbm_step), the slabs stepped then exchanged (lbm_step + lbm_halo_pack, copies,
    lbm_halo_unpack), and the slabs with the exchange overlapped by the interior planes
    (lbm_slab_step_begin, copies, lbm_slab_step_end).  On one GPU nothing crosses a link, so this
    measures what the decomposition itself costs; MLUPS count the owned cells."""
    from lattice_boltzmann_cfd_d3q19_gb300 import slab as S
    flags = porous_flags(n)
    N = n ** 3
    stream = torch.cuda.current_stream()

    def setup(ctx, nz, fl):
        B.lbm_set_stream(ctx, stream.cuda_stream)
        B.lbm_set_flags(ctx, fl)
        B.lbm_set_body_force(ctx, 1e-6, 0.0, 0.0)
        M = n * n * nz
        B.lbm_set_equilibrium(ctx, torch.ones(M, dtype=torch.float32, device="cuda"),
                              torch.zeros(3 * M, dtype=torch.float32, device="cuda"))

    def timed(step):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    out = {"slabs": world, "halo_bytes_per_slab_and_step": 2 * 5 * n * n * 4}
    ctx = B.lbm_create(n, n, n, 0.7, B.LAYOUT_STREAM, B.STREAMING_AB)
    try:
        setup(ctx, n, flags)
        ms = timed(lambda: B.lbm_step(ctx, 1))
    finally:
        B.lbm_destroy(ctx)
    out["unsliced"] = {"ms_per_lbm_step": round(ms, 4), "mlups": round(N / ms / 1e3, 1)}
    slabs = [S.slab_of(n, r, world) for r in range(world)]
    ctxs = []
    try:
        for sl in slabs:
            c = B.lbm_create(n, n, sl.local_nz, 0.7, B.LAYOUT_STREAM, B.STREAMING_AB)
            ctxs.append(c)
            B.lbm_set_ghost_planes(c, True)
            setup(c, sl.local_nz, S.local_slice(flags, sl, n, n))
        eng = [S.LibraryEngine(c) for c in ctxs]
        recv = [(e.halo_like(), e.halo_like()) for e in eng]  # (from below, from above)

        def swap(packed):
            for r, sl in enumerate(slabs):
                recv[r][0].copy_(packed[sl.below][1])
                recv[r][1].copy_(packed[sl.above][0])

        def serial():
            for e in eng:
                e.step1()
            swap([e.pack() for e in eng])
            for e, (fb, fa) in zip(eng, recv):
                e.unpack(fb, fa)

        def overlapped():
            swap([e.begin() for e in eng])
            for e, (fb, fa) in zip(eng, recv):
                e.end(fb, fa)

        for name, fn in (("slabs_serial", serial), ("slabs_overlapped", overlapped)):
            ms = timed(fn)
            out[name] = {"ms_per_lbm_step": round(ms, 4), "mlups": round(N / ms / 1e3, 1)}
    finally:
        for c in ctxs:
            B.lbm_destroy(c)
    return out


def cpu_description():
    """Host CPU for the CPU baseline: architecture, model (x86 'model name', or the Arm
    implementer/part codes) and logical CPU count."""
    import platform
    model = None
    try:
        info = {}
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k, _, v = line.partition(":")
                info.setdefault(k.strip(), v.strip())
        model = info.get("model name") or (
            f"implementer {info['CPU implementer']} part {info['CPU part']}"
            if "CPU part" in info else None)
    except OSError:
        pass
    return {"machine": platform.machine(), "model": model, "logical_cpus": os.cpu_count()}


def cpu_baseline(n=512, ny_sample=16, target_s=15.0):
    """The CPU oracle, as it is, on a bounded sample of the porous workload: a 512 x ny_sample x
    512 slab of the same flags (periodic), same tau and body force."""
    import oracle
    flags = porous_flags(n).reshape(n, n, n)
    sub = np.ascontiguousarray(flags[:, :ny_sample, :]).reshape(-1)
    Ns = n * ny_sample * n
    P = oracle.Problem(n, ny_sample, n, 0.7, flags=sub, g=(1e-6, 0, 0))
    f = oracle.equilibrium_field(*wl.uniform_fields(Ns))
    t0 = time.perf_counter()
    f, _ = P.step_ab(f, 1)
    one = time.perf_counter() - t0
    steps = int(max(1, min(200, target_s / max(one, 1e-3))))
    t0 = time.perf_counter()
    P.step_ab(f, steps)
    dt = time.perf_counter() - t0
    cores = oracle.max_threads()  # before the one-thread run below sets the thread count
    # one thread, on a thinner slab of the same flags (a few seconds)
    ny1 = 2
    sub1 = np.ascontiguousarray(flags[:, :ny1, :]).reshape(-1)
    N1 = n * ny1 * n
    P1 = oracle.Problem(n, ny1, n, 0.7, flags=sub1, g=(1e-6, 0, 0), threads=1)
    f1 = oracle.equilibrium_field(*wl.uniform_fields(N1))
    t0 = time.perf_counter()
    P1.step_ab(f1, 4)
    dt1 = time.perf_counter() - t0
    return {"value": round(Ns * steps / dt / 1e6, 3), "unit": UNIT, "cores": cores,
            "kind": "oracle", "cpu": cpu_description(),
            "sample": f"{n}x{ny_sample}x{n} slab of the porous 512^3 flags, periodic, {steps} steps "
                      f"({dt:.1f} s), fp64 two-lattice oracle",
            "single_thread": {"value": round(N1 * 4 / dt1 / 1e6, 3), "unit": UNIT, "cores": 1,
                              "sample": f"{n}x{ny1}x{n} slab, 4 steps ({dt1:.1f} s)"}}


def variant_specs():
    """The variant workloads of the JSON line: name -> (edge, scheme, options of variant())."""
    specs = {}
    for m in (128, 512):
        for s in ("AA", "AB"):
            specs[f"{s}_{m}^3_periodic"] = (m, s, {})
    for lay in ("bundle", "collision"):
        for s in ("AA", "AB"):
            specs[f"{s}_128^3_periodic_{lay}_layout"] = (128, s, {"layout": lay})
    for s in ("AA", "AB"):
        specs[f"{s}_128^3_sphere_inlet_outlet"] = (128, s, {"sphere": True})
    specs["AA_256^3_lid_driven_cavity"] = (256, "AA", {"cavity": True})
    for s in ("AA", "AB"):
        specs[f"{s}_512^3_periodic_fp16_storage"] = (512, s, {"fp16": True})
    specs["AA_512^3_porous_fp16_storage"] = (512, "AA", {"fp16": True, "porous": True})
    specs["AB_512^3_porous_2_z_slabs_one_gpu"] = (512, "AB", {"slabs": 2})
    return specs


def run_variant(B, torch, m, s, steps, warmup, **kw):
    if "slabs" in kw:
        return slab_variant(B, torch, m, kw["slabs"], steps=steps, warmup=warmup)
    return variant(B, torch, m, s, steps=steps, warmup=warmup, **kw)


def run_variants_only(args):
    """--variant: the named variant workloads alone (a command for profiling captures), one JSON
    line each; --variant-size replaces their edge."""
    specs = variant_specs()
    for name in args.variant:
        if name not in specs:
            raise SystemExit(f"unknown variant {name!r}; known: {', '.join(specs)}")
    import torch
    from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
    B.load()
    for name in args.variant:
        m, s, kw = specs[name]
        m = args.variant_size or m
        res = run_variant(B, torch, m, s, args.steps, args.warmup, **kw)
        print(json.dumps({"variant": name, "edge": m, **res}), flush=True)


def e2e_run(B, torch, n, steps, flags):
    """Through the public API with host buffers: load the state from pinned host memory, run the
    steps reading the drag force back after each, read rho and u back to pinned host memory."""
    N = n ** 3
    ctx = B.lbm_create(n, n, n, 0.7, B.LAYOUT_STREAM, B.STREAMING_AA)
    try:
        B.lbm_set_flags(ctx, flags)
        B.lbm_set_body_force(ctx, 1e-6, 0, 0)
        f_host = torch.empty((19, N), dtype=torch.float32, pin_memory=True)
        for q in range(19):
            f_host[q].fill_(1 / 3 if q == 0 else 1 / 18 if q <= 6 else 1 / 36)
        rho_host = torch.empty(N, dtype=torch.float32, pin_memory=True)
        u_host = torch.empty(3 * N, dtype=torch.float32, pin_memory=True)
        B.lbm_set_stream(ctx, torch.cuda.current_stream().cuda_stream)
        # warm-up of the same sequence
        B.lbm_set_populations(ctx, f_host)
        B.lbm_step(ctx, 2)
        B.lbm_force_momentum_exchange(ctx)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        B.lbm_set_populations(ctx, f_host)
        for _ in range(steps):
            B.lbm_step(ctx, 2)
            B.lbm_force_momentum_exchange(ctx)
        B.lbm_macroscopic(ctx, rho_host, u_host)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        B.lbm_destroy(ctx)
    return {"value": round(N * 2 * steps / dt / 1e6, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(19 * N * 4 / steps),
            "d2h_bytes_per_step": int((4 * N * 4 + 24 * steps) / steps),
            "what": "per step: 2 LBM steps + drag force read back; the population upload and the "
                    "rho/u read-back are spread over the steps"}


def run_ours(args):
    import torch
    from lattice_boltzmann_cfd_d3q19_gb300 import binding as B

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    B.load()
    n, tau, g = args.size, 0.7, (1e-6, 0.0, 0.0)
    N = n ** 3
    log(f"[bench] rank {rank}: building porous {n}^3 workload")
    ctx, flags = make_porous_context(B, torch, n, tau, g)
    n_fluid = int(np.count_nonzero(flags == wl.FLUID))
    sampler = ClockSampler(local) if rank == 0 else None
    try:
        ms, launches, prof, clocks, step_ms = timed_steps(B, torch, ctx, args.steps, args.warmup,
                                                          sampler=sampler, world=world)
    finally:
        B.lbm_destroy(ctx)
    max_s = reduce_max(ms / 1e3, world, device="cuda")
    value = whole_job_mlups(N * 2, args.steps, world, max_s)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    # dominant kernel by total time in the timed region
    step_kernels = {k: v for k, v in prof.items() if k != "force_reduce"}
    dom = max(step_kernels, key=lambda k: step_kernels[k][1])
    cnt, tot = step_kernels[dom]
    per_launch_s = tot / cnt / 1e3
    alg = algorithmic_bytes(N)
    achieved = alg / per_launch_s / 1e9
    achieved_fluid = fluid_bytes(N, n_fluid) / per_launch_s / 1e9
    traffic_per_cell = recorded_traffic(dom)
    kernels = {k: {"launches": c, "avg_ms": round(t / c, 4),
                   "GB/s": round(alg / (t / c / 1e3) / 1e9, 1) if k != "force_reduce" else None}
               for k, (c, t) in prof.items()}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 4),
        # each timed step alone (CUDA events between steps, rank 0): the median of the runs
        # with their spread
        "step_ms": {"median": round(statistics.median(step_ms), 4), "min": round(min(step_ms), 4),
                    "max": round(max(step_ms), 4), "runs": len(step_ms)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(workload_config(n, tau, g, n_fluid / N),
                       fluid_mlups=round(value * n_fluid / N, 1)),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": alg,
                     "bytes_rule": "153 B per cell update (19 x 4 B read + 19 x 4 B written + "
                                   "1 B flag), every cell",
                     "fluid_only": {"achieved": round(achieved_fluid, 1),
                                    "frac": round(achieved_fluid / peak, 4),
                                    "rule": "152 B per FLUID cell + 1 B flag per cell"},
                     "traffic": (round(traffic_per_cell * N) if traffic_per_cell else None),
                     "traffic_source": "profiles/ncu_traffic.txt (per-cell DRAM bytes of a 256^3 "
                                       "capture, scaled by cells)"},
        "kernels": kernels,
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if not args.no_variants:
        log("[bench] variants")
        out["variants"] = {name: run_variant(B, torch, m, s, 10, 3, **kw)
                           for name, (m, s, kw) in variant_specs().items()}
    if not args.no_e2e:
        log("[bench] e2e")
        out["e2e"] = e2e_run(B, torch, n, args.steps, flags)
    if not args.no_cpu_baseline:
        log("[bench] cpu baseline")
        out["cpu_baseline"] = cpu_baseline()
    print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step is 2 oracle time steps on a bounded sample
    (a 512 x 8 x 512 slab of the porous workload)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    n, ny_s = 512, 8
    flags = wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512).reshape(n, n, n)
    sub = np.ascontiguousarray(flags[:, :ny_s, :]).reshape(-1)
    Ns = n * ny_s * n
    P = oracle.Problem(n, ny_s, n, 0.7, flags=sub, g=(1e-6, 0, 0))
    f = oracle.equilibrium_field(*wl.uniform_fields(Ns))
    for _ in range(args.warmup):
        f, _ = P.step_ab(f, 2)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        f, _ = P.step_ab(f, 2)
    dt = time.perf_counter() - t0
    value = Ns * 2 * args.steps / dt / 1e6
    sample = f"{n}x{ny_s}x{n} slab of the porous 512^3 flags, periodic, 2 oracle steps per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(n, 0.7, (1e-6, 0.0, 0.0),
                                       float((flags == wl.FLUID).mean())),
                       sample=sample),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "cpu": cpu_description(), "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", action="append", default=[],
                    help="run only this variant workload (repeatable; names as in the JSON "
                         "line's 'variants'), one JSON line each: for profiling captures")
    ap.add_argument("--variant-size", type=int, default=0,
                    help="edge for --variant instead of the variant's own")
    ap.add_argument("--size", type=int, default=512,
                    help="edge of the porous workload (512 is the benchmark; smaller sizes are "
                         "for profiling captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.variant:
        run_variants_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
