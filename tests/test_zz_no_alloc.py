"""The entry point that allocates nothing, against the context-based force it mirrors and against
the oracle.

lbm_force_momentum_exchange_noalloc serves callers that cannot call cudaMalloc: plug-ins whose
host application owns all device memory through its own pool, and tools that must not grow the
footprint of a process they are embedded in.  Its working memory is a fixed array in the
library's static device memory.  Here it must give the same force as lbm_set_populations +
lbm_step(1) + lbm_force_momentum_exchange on the same state, and as the oracle's two-lattice step
with the force of that step, on two calls in a row (the second call reuses the array the first
one left behind).  This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

# the force tolerance the other parity tests use: relative to the force scale
REL = 1e-4


def make_state(nx, ny, nz, seed):
    r = np.random.default_rng(seed)
    N = nx * ny * nz
    rho = 1 + r.uniform(-0.02, 0.02, N)
    u = r.uniform(-0.04, 0.04, (3, N))
    u[0] += 0.03
    f = oracle.equilibrium_field(rho, u) * (1 + 5e-3 * r.uniform(-1, 1, (19, N)))
    return f.astype(np.float32)


def context_force(f, flags, n, faces, tau, g):
    ctx = B.lbm_create(*n, tau)
    try:
        B.lbm_set_flags(ctx, flags)
        B.lbm_set_faces(ctx, *faces)
        B.lbm_set_body_force(ctx, *g)
        B.lbm_set_populations(ctx, f)
        B.lbm_step(ctx, 1)
        return B.lbm_force_momentum_exchange(ctx)
    finally:
        B.lbm_destroy(ctx)


def oracle_force(f, flags, n, faces, tau, g):
    P = oracle.Problem(*n, tau, flags=flags, faces=faces, g=g)
    _, F = P.step_ab(f.astype(np.float64), 1, want_force=True)
    return F


CASES = [
    # grid, faces, geometry, tau, g
    ((40, 30, 28), (0, 0, 0), "sphere", 0.7, (0.0, 0.0, 0.0)),
    ((33, 21, 17), (1, 0, 0), "porous", 0.62, (2e-5, -1e-5, 0.0)),
    # an INLET layer on an OPEN x face: inlet cells are neither collided nor bounce-back partners
    ((36, 20, 18), (1, 0, 0), "sphere_inlet", 0.6, (1e-5, 0.0, 0.0)),
]


def case_flags(n, geom):
    if geom == "sphere":
        return wl.sphere_flags(*n, (14, 15, 14), 6, inlet_x0=False)
    if geom == "sphere_inlet":
        return wl.sphere_flags(*n, (12, 10, 9), 5, inlet_x0=True)
    return wl.porous_flags(*n, 0.2, 3, seed=77)


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_noalloc_force_matches_context_force_and_oracle_twice(ci):
    n, faces, geom, tau, g = CASES[ci]
    flags = case_flags(n, geom)
    if geom == "sphere_inlet":
        assert (flags == wl.INLET).any()
    f = make_state(*n, 500 + ci)
    F_ref = context_force(f, flags, n, faces, tau, g)
    F_orc = oracle_force(f, flags, n, faces, tau, g)
    f_dev = torch.from_numpy(f.reshape(-1).copy()).cuda()
    flags_dev = torch.from_numpy(flags.copy()).cuda()
    scale = float(np.abs(F_orc).max())
    assert scale > 0
    assert np.abs(F_ref - F_orc).max() <= REL * scale, (F_ref, F_orc)
    for _ in range(2):
        F = B.lbm_force_momentum_exchange_noalloc(f_dev, flags_dev, *n, faces=faces, tau=tau, g=g)
        assert np.abs(F - F_ref).max() <= REL * scale, (F, F_ref)
        assert np.abs(F - F_orc).max() <= REL * scale, (F, F_orc)


def test_noalloc_rejects_moving_wall_flags_and_leaves_F_unchanged():
    n = (12, 10, 8)
    N = n[0] * n[1] * n[2]
    flags = wl.sphere_flags(*n, (6, 5, 4), 2, inlet_x0=False)
    flags[flags == wl.SOLID] = wl.MOVING_WALL
    f_dev = torch.from_numpy(make_state(*n, 9).reshape(-1).copy()).cuda()
    flags_dev = torch.from_numpy(flags).cuda()
    F = (ctypes.c_double * 3)(11.0, 22.0, 33.0)
    rc = B.load().lbm_force_momentum_exchange_noalloc(
        f_dev.data_ptr(), flags_dev.data_ptr(), *n, 0, 0, 0, 0.6, 0.0, 0.0, 0.0,
        ctypes.addressof(F), None)
    assert rc == B.EINVAL
    assert "0, 1 or 2" in B.lbm_last_error()
    assert list(F) == [11.0, 22.0, 33.0]
    assert f_dev.numel() == 19 * N
    # a valid call right after the rejected one is not disturbed by its error word
    flags_dev = torch.from_numpy(np.where(flags == wl.MOVING_WALL, wl.SOLID, flags)
                                 .astype(np.uint8)).cuda()
    B.lbm_force_momentum_exchange_noalloc(f_dev, flags_dev, *n, tau=0.6)


def test_noalloc_rejects_grids_beyond_its_scratch():
    dims = (257, 256, 256)
    N = dims[0] * dims[1] * dims[2]
    f = torch.zeros(19 * N, dtype=torch.float32, device="cuda")
    flags = torch.zeros(N, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.LbmError) as ei:
        B.lbm_force_momentum_exchange_noalloc(f, flags, *dims)
    assert ei.value.code == B.EINVAL and "scratch limit" in str(ei.value)
    del f, flags
    torch.cuda.empty_cache()
