"""Writes the full-length oracle fixtures ``full_<name>.npz`` used by tests/test_gpu_full_length.py.

Runs only the CPU oracle (``oracle/``) on the seeded inputs of ``workloads.py``; no value here comes
from the CUDA library.  Three workloads, at their full sizes and step counts:

  * taylor_green_128 -- periodic 128^3, tau 0.6, Taylor-Green u0 = 0.05, rho = 1, f = f_eq, 1000
    steps (the 128^3 periodic case of "GPU lattice Boltzmann: streaming layout and performance",
    results table; the Taylor-Green vortex is a validation case of "PortLBM ...", §5);
  * sphere_128 -- 128^3, SOLID sphere r = 16 at (40, 64, 64), INLET layer x = 0 at
    f_eq(1, (0.05, 0, 0)), x OPEN (zero-gradient), y/z periodic, tau 0.56, f = f_eq(1, u_in),
    2000 steps, momentum-exchange force of the last step (the sphere 128^3 case of the same table);
  * porous_512 -- 512^3, 3^3 solid blobs to a solid fraction of 0.30 (seed 1005), periodic,
    body acceleration g = (1e-6, 0, 0) with Guo forcing, tau 0.7, rho = 1, u = 0, 500 steps, force
    of the last step (porous-medium runs of "PortLBM ...", §5).

Each fixture holds, for a seeded sample of FLUID cells (sorted cell indices n = x + nx (y + ny z)):
the natural populations f[19, S] after the last step, rho[S] and u[3, S] (with the half-force
shift of Guo forcing) in float64, and the force triple of the last step; ``meta`` (JSON) records
the workload, step count, sample seed and the hash of the oracle source (comments and white space
dropped) that produced it.

Both sides start from the same float32 state: f_eq from the oracle in float64, rounded to float32
(the GPU library stores fp32); the oracle runs on those rounded values widened back to float64.

Usage:  python tests/golden/make_full_length_goldens.py [--only NAME ...] [--out DIR] [--threads T]
The porous 512^3 run holds two fp64 lattices (41 GB of host memory) and takes about 17 minutes on
16 cores; the 128^3 runs a few minutes each.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl  # noqa: E402

SAMPLE = 65536          # random FLUID cells per workload
NAMES = ("taylor_green_128", "sphere_128", "porous_512")
SAMPLE_SEED = {"taylor_green_128": 2003, "sphere_128": 2004, "porous_512": 2005}


def oracle_source_hash() -> str:
    """sha256 of the oracle's C++ source with comments and white space removed, so that a fixture
    is known to be stale exactly when the oracle's code changes."""
    with open(os.path.join(ROOT, "oracle", "d3q19_oracle.cpp"), encoding="utf-8") as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"\s+", "", src)
    return hashlib.sha256(src.encode()).hexdigest()


def spec(name: str) -> dict:
    """Grid, relaxation time, flags, faces, inlet, body acceleration, step count and the uniform
    initial state (rho, u) or None for a Taylor-Green field."""
    if name == "taylor_green_128":
        n = 128
        return dict(dims=(n, n, n), tau=0.6, flags=np.zeros(n ** 3, np.uint8), faces=(0, 0, 0),
                    inlet=(1.0, 0.0, 0.0, 0.0), g=(0.0, 0.0, 0.0), steps=1000, force=False,
                    uniform=None, tg_u0=0.05)
    if name == "sphere_128":
        n, u_in = 128, 0.05
        return dict(dims=(n, n, n), tau=0.56,
                    flags=wl.sphere_flags(n, n, n, (40, 64, 64), 16, inlet_x0=True),
                    faces=(1, 0, 0), inlet=(1.0, u_in, 0.0, 0.0), g=(0.0, 0.0, 0.0),
                    steps=2000, force=True, uniform=(1.0, (u_in, 0.0, 0.0)), tg_u0=None)
    if name == "porous_512":
        n = 512
        return dict(dims=(n, n, n), tau=0.7,
                    flags=wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512),
                    faces=(0, 0, 0), inlet=(1.0, 0.0, 0.0, 0.0), g=(1e-6, 0.0, 0.0),
                    steps=500, force=True, uniform=(1.0, (0.0, 0.0, 0.0)), tg_u0=None)
    raise KeyError(name)


def initial_f32_columns(s: dict):
    """For a uniform initial state: the 19 float32 populations shared by every cell.  None for a
    Taylor-Green field (use initial_f32_field)."""
    if s["uniform"] is None:
        return None
    rho, u = s["uniform"]
    return oracle.equilibrium(rho, u).astype(np.float32)


def initial_f32_field(s: dict) -> np.ndarray:
    """float32 f[19, N] of the Taylor-Green initial state (f = f_eq in float64, then rounded)."""
    nx, ny, nz = s["dims"]
    rho, u = wl.taylor_green(nx, ny, nz, s["tg_u0"])
    return oracle.equilibrium_field(rho, u).astype(np.float32)


def sample_cells(name: str, s: dict) -> np.ndarray:
    """Sorted FLUID cell indices: SAMPLE drawn uniformly without replacement (PCG64, per-workload
    seed), plus, for the sphere, every fluid cell within two cells of the sphere's surface and a
    regular subsample of the layers next to the inlet and the outlet."""
    flags = s["flags"]
    fluid = np.flatnonzero(flags == wl.FLUID)
    g = wl.rng(SAMPLE_SEED[name])
    cells = g.choice(fluid, size=SAMPLE, replace=False)
    if name == "sphere_128":
        nx, ny, nz = s["dims"]
        x, y, z = wl.coords(nx, ny, nz)
        shell = (x - 40) ** 2 + (y - 64) ** 2 + (z - 64) ** 2 <= 18 ** 2
        faces = np.isin(x, (1, 2, nx - 2, nx - 1)) & (y % 4 == 1) & (z % 4 == 2)
        extra = np.flatnonzero((shell | faces) & (flags == wl.FLUID))
        cells = np.concatenate([cells, extra])
    return np.unique(cells).astype(np.int64)


def run(name: str, out_dir: str, threads: int = 0) -> str:
    s = spec(name)
    nx, ny, nz = s["dims"]
    N = nx * ny * nz
    t0 = time.time()
    cols = initial_f32_columns(s)
    if cols is None:
        f = initial_f32_field(s).astype(np.float64)
    else:
        f = np.empty((19, N), np.float64)
        for q in range(19):
            f[q].fill(float(cols[q]))
    P = oracle.Problem(nx, ny, nz, s["tau"], flags=s["flags"], faces=s["faces"], inlet=s["inlet"],
                       g=s["g"], threads=threads)
    f, force = P.step_ab(f, s["steps"], want_force=True, inplace=True)
    rho, u = P.macroscopic(f)
    cells = sample_cells(name, s)
    elapsed = time.time() - t0
    meta = dict(workload=name, dims=list(s["dims"]), tau=s["tau"], steps=s["steps"],
                faces=list(s["faces"]), inlet=list(s["inlet"]), g=list(s["g"]),
                sample_seed=SAMPLE_SEED[name], sample=int(cells.size),
                oracle_hash=oracle_source_hash(), oracle_threads=oracle.max_threads(),
                seconds=round(elapsed, 1), machine=platform.machine(),
                force_checked=bool(s["force"]))
    path = os.path.join(out_dir, f"full_{name}.npz")
    np.savez_compressed(path, cells=cells, f=np.ascontiguousarray(f[:, cells]),
                        rho=rho[cells], u=np.ascontiguousarray(u[:, cells]), force=force,
                        meta=np.array(json.dumps(meta)))
    print(f"{name}: {s['steps']} steps, {cells.size} cells, {elapsed:.0f} s -> {path}",
          flush=True)
    return path


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", nargs="*", default=list(NAMES))
    ap.add_argument("--out", default=HERE)
    ap.add_argument("--threads", type=int, default=0)
    a = ap.parse_args()
    os.makedirs(a.out, exist_ok=True)
    for name in a.only:
        run(name, a.out, a.threads)


if __name__ == "__main__":
    main()
