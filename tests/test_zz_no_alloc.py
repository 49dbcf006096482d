"""The entry point that allocates nothing, against the context-based force it mirrors.

lbm_force_momentum_exchange_noalloc serves callers that cannot call cudaMalloc (for instance code
running while a CUDA graph is captured on its stream, or a plug-in whose host owns all device
memory): its working memory is a fixed array in the library's static device memory.  Here it
must give the same force as lbm_set_populations + lbm_step(1) + lbm_force_momentum_exchange on
the same state, on two calls in a row (the second call reuses the array the first one left
behind).  This file is collected last so that a run stopping at the first failure has already
run every other test.
"""
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


CASES = [
    # grid, faces, geometry, tau, g
    ((40, 30, 28), (0, 0, 0), "sphere", 0.7, (0.0, 0.0, 0.0)),
    ((33, 21, 17), (1, 0, 0), "porous", 0.62, (2e-5, -1e-5, 0.0)),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_noalloc_force_matches_context_force_twice(ci):
    n, faces, geom, tau, g = CASES[ci]
    N = n[0] * n[1] * n[2]
    if geom == "sphere":
        flags = wl.sphere_flags(*n, (14, 15, 14), 6, inlet_x0=False)
    else:
        flags = wl.porous_flags(*n, 0.2, 3, seed=77)
    f = make_state(*n, 500 + ci)
    F_ref = context_force(f, flags, n, faces, tau, g)
    f_dev = torch.from_numpy(f.reshape(-1).copy()).cuda()
    flags_dev = torch.from_numpy(flags.copy()).cuda()
    scale = float(np.abs(F_ref).max())
    assert scale > 0
    for _ in range(2):
        F = B.lbm_force_momentum_exchange_noalloc(f_dev, flags_dev, *n, faces=faces, tau=tau, g=g)
        assert np.abs(F - F_ref).max() <= REL * scale, (F, F_ref)


def test_noalloc_rejects_grids_beyond_its_scratch():
    f = torch.zeros(19, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.LbmError) as ei:
        B.lbm_force_momentum_exchange_noalloc(f, flags, 257, 256, 256)
    assert ei.value.code == B.EINVAL and "scratch limit" in str(ei.value)
