"""Full-length parity: the CUDA library, through the C ABI, against fp64 oracle fixtures of the three
large workloads at their stated sizes and step counts.

  * periodic Taylor-Green 128^3, 1000 steps: AA and A-B in the stream, bundle and collision layouts
    (the periodic 128^3 case of "GPU lattice Boltzmann: streaming layout and performance", results
    table);
  * sphere 128^3 with equilibrium inlet, zero-gradient outlet and bounce-back sphere, 2000 steps,
    with the momentum-exchange drag: AA and A-B, stream layout (the sphere 128^3 case of the same
    table);
  * porous medium 512^3 under a Guo body force, 500 steps, with the force on the solids: AA and
    A-B, stream layout, the AA run in the benchmark's launch configuration ("PortLBM ...", §5).

The fixtures (tests/golden/full_*.npz) are written by tests/golden/make_full_length_goldens.py,
which runs only the CPU oracle.  Each run here is compared on the fixture's sampled FLUID cells:
max |f_gpu - f_oracle| <= 1e-5 (the method's fp32 bar, rho ~ 1), rho and u within 1e-5, the force
within 1e-4 of max(1, |F|).  The measured differences are printed (pytest -s shows them).
"""
import json
import os
import sys

import numpy as np
import pytest

from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
from lbm_harness import LAYOUTS, SCHEMES, TOL_F

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_full_length_goldens as G  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

TOL_FORCE = 1e-4  # relative to max(1, |F|)


def load_fixture(name):
    path = os.path.join(HERE, "golden", f"full_{name}.npz")
    assert os.path.exists(path), f"missing fixture {path}"
    z = np.load(path)
    meta = json.loads(str(z["meta"]))
    assert meta["oracle_hash"] == G.oracle_source_hash(), "fixture is stale: regenerate it"
    return z, meta


_specs = {}


def workload(name):
    if name not in _specs:
        _specs[name] = G.spec(name)
    return _specs[name]


def run_gpu(name, layout, scheme):
    """Runs the workload's full step count; returns sampled f, rho, u (float64) and the force."""
    s = workload(name)
    z, meta = load_fixture(name)
    nx, ny, nz = s["dims"]
    N = nx * ny * nz
    assert meta["steps"] == s["steps"] and meta["dims"] == [nx, ny, nz]
    cols = G.initial_f32_columns(s)
    if cols is None:
        f0 = torch.from_numpy(G.initial_f32_field(s)).cuda()
    else:
        f0 = torch.from_numpy(cols).cuda()[:, None].expand(19, N).contiguous()
    ctx = B.lbm_create(nx, ny, nz, s["tau"], LAYOUTS[layout], SCHEMES[scheme])
    try:
        B.lbm_set_flags(ctx, torch.from_numpy(s["flags"]).cuda())
        B.lbm_set_faces(ctx, *s["faces"])
        B.lbm_set_inlet(ctx, *s["inlet"])
        B.lbm_set_body_force(ctx, *s["g"])
        B.lbm_set_populations(ctx, f0)
        del f0
        B.lbm_step(ctx, s["steps"])
        assert B.lbm_check_finite(ctx)
        F = B.lbm_force_momentum_exchange(ctx)
        cells = torch.from_numpy(z["cells"]).cuda()
        f = torch.empty((19, N), dtype=torch.float32, device="cuda")
        B.lbm_get_populations(ctx, f)
        fs = f[:, cells].cpu().numpy().astype(np.float64)
        del f
        rho = torch.empty(N, dtype=torch.float32, device="cuda")
        u = torch.empty((3, N), dtype=torch.float32, device="cuda")
        B.lbm_macroscopic(ctx, rho, u)
        rs = rho[cells].cpu().numpy().astype(np.float64)
        us = u[:, cells].cpu().numpy().astype(np.float64)
        del rho, u
    finally:
        B.lbm_destroy(ctx)
        torch.cuda.empty_cache()
    return z, fs, rs, us, np.asarray(F, np.float64)


def check(name, layout, scheme):
    z, fs, rs, us, F = run_gpu(name, layout, scheme)
    df = float(np.abs(fs - z["f"]).max())
    dr = float(np.abs(rs - z["rho"]).max())
    du = float(np.abs(us - z["u"]).max())
    Fo = z["force"]
    scale = max(1.0, float(np.abs(Fo).max()))
    dF = float(np.abs(F - Fo).max()) / scale
    print(f"\nfull-length parity {name} {scheme} {layout}: cells {z['cells'].size}, "
          f"max|df| {df:.3e}, max|drho| {dr:.3e}, max|du| {du:.3e}, force {F.tolist()} "
          f"vs oracle {Fo.tolist()} (rel {dF:.3e})")
    assert df <= TOL_F, df
    assert dr <= TOL_F, dr
    assert du <= TOL_F, du
    assert dF <= TOL_FORCE, (F, Fo)


@pytest.mark.parametrize("scheme", ["AA", "AB"])
@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
def test_taylor_green_128_1000_steps(layout, scheme):
    check("taylor_green_128", layout, scheme)


@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_sphere_128_2000_steps(scheme):
    check("sphere_128", "stream", scheme)


@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_porous_512_500_steps(scheme):
    check("porous_512", "stream", scheme)
