"""The library's side of the z-slab decomposition on one GPU: ghost planes (lbm_set_ghost_planes),
the halo kernels (lbm_halo_pack / lbm_halo_unpack) and the step with the exchange overlapped by the
interior planes (lbm_slab_step_begin / lbm_slab_step_end).  Several slab contexts live in one
process and the host swaps their halo buffers between steps, in order (no kernel waits on
another).  The slabs together must give the unsliced context's populations bit for bit (the same
kernels on the same values) and its force up to the grouping of the fp64 sums ("Disaggregated
Design for GPU-Based Volumetric Data Structures", "Improving LBM Scalability": each partition
exchanges its boundary data with its neighbours every step; "Disaggregation on a Dense Domain":
the exchange overlaps the voxels that need no neighbour data)."""
import numpy as np
import pytest

from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
from lattice_boltzmann_cfd_d3q19_gb300 import slab as S
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl
from lbm_harness import LAYOUTS, FP16, random_state

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

TAU, G, INLET = 0.62, (2e-5, -1e-5, 1e-5), (1.0, 0.04, 0.0, 0.0)


WALL = (0.03, -0.01, 0.02)


def global_problem(nx, ny, nz, seed, moving):
    """Random solids (a third of them moving walls when `moving`), an inlet layer on x = 0."""
    r = np.random.default_rng(seed)
    N = nx * ny * nz
    flags = (r.uniform(size=N) < 0.15).astype(np.uint8)
    if moving:
        flags[(flags == wl.SOLID) & (r.uniform(size=N) < 0.33)] = wl.MOVING_WALL
    x, _, _ = wl.coords(nx, ny, nz)
    flags[x == 0] = wl.INLET
    f0 = random_state(N, seed + 1).astype(np.float32)
    return flags, f0


def make_ctx(nx, ny, nz, layout, flags, pairs):
    ctx = B.lbm_create(nx, ny, nz, TAU, {**LAYOUTS, **FP16}[layout], B.STREAMING_AB)
    B.lbm_set_cell_pairs(ctx, pairs)
    B.lbm_set_flags(ctx, flags)
    B.lbm_set_faces(ctx, B.OPEN, B.PERIODIC, B.PERIODIC)
    B.lbm_set_inlet(ctx, *INLET)
    B.lbm_set_body_force(ctx, *G)
    B.lbm_set_wall_velocity(ctx, *WALL)
    return ctx


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("moving", [False, True])
@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("layout", ["stream", "bundle", "collision", "stream_fp16"])
@pytest.mark.parametrize("nz, world", [(12, 2), (13, 3), (4, 4), (6, 3)])
def test_slabs_equal_the_unsliced_context(nz, world, layout, pairs, moving, overlap):
    """With moving walls the slabs also have special cells (boundary kernel), some of them next
    to a ghost plane.  (4, 4): every slab owns one plane (no interior); (6, 3): two (both are
    boundary planes)."""
    nx, ny, steps = 10, 8, 6
    flags, f0 = global_problem(nx, ny, nz, 70 + nz, moving)
    ref = make_ctx(nx, ny, nz, layout, flags, pairs)
    try:
        B.lbm_set_populations(ref, torch.from_numpy(f0.reshape(-1).copy()).cuda())
        B.lbm_step(ref, steps)
        want = np.zeros((19, nx * ny * nz), np.float32)
        B.lbm_get_populations(ref, want)
        F_want = B.lbm_force_momentum_exchange(ref)
    finally:
        B.lbm_destroy(ref)
    slabs = [S.slab_of(nz, r, world) for r in range(world)]
    ctxs = []
    try:
        for s in slabs:
            c = make_ctx(nx, ny, s.local_nz, layout, S.local_slice(flags, s, nx, ny), pairs)
            ctxs.append(c)
            B.lbm_set_ghost_planes(c, True)
            B.lbm_set_populations(c, torch.from_numpy(S.local_slice(f0, s, nx, ny).reshape(-1)).cuda())
        eng = [S.LibraryEngine(c) for c in ctxs]
        for _ in range(steps):
            if overlap:
                packed = [e.begin() for e in eng]  # (lo, hi) per slab; interiors still running
                for r, e in enumerate(eng):
                    s = slabs[r]
                    e.end(packed[s.below][1], packed[s.above][0])
            else:
                for e in eng:
                    e.step1()
                packed = [e.pack() for e in eng]  # (lo, hi) per slab
                for r, e in enumerate(eng):
                    s = slabs[r]
                    e.unpack(packed[s.below][1], packed[s.above][0])
        got, F = [], np.zeros(3)
        for s, c in zip(slabs, ctxs):
            loc = np.zeros((19, nx * ny * s.local_nz), np.float32)
            B.lbm_get_populations(c, loc)
            got.append(S.owned_part(loc, s, nx, ny))
            F += B.lbm_force_momentum_exchange(c)
    finally:
        for c in ctxs:
            B.lbm_destroy(c)
    got = np.concatenate(got, axis=1)
    fluid = flags == wl.FLUID
    assert np.array_equal(got[:, fluid], want[:, fluid])
    assert np.abs(F - F_want).max() <= 1e-4 * max(1.0, float(np.abs(F_want).max())), (F, F_want)


def test_ghost_plane_rules():
    ctx = B.lbm_create(8, 6, 5, 0.6, B.LAYOUT_STREAM, B.STREAMING_AA)
    try:
        with pytest.raises(B.LbmError) as ei:
            B.lbm_set_ghost_planes(ctx, True)
        assert ei.value.code == B.EINVAL and "A-B" in str(ei.value)
    finally:
        B.lbm_destroy(ctx)
    ctx = B.lbm_create(8, 6, 5, 0.6, B.LAYOUT_STREAM, B.STREAMING_AB)
    try:
        B.lbm_set_ghost_planes(ctx, True)
        with pytest.raises(B.LbmError) as ei:
            B.lbm_set_faces(ctx, B.PERIODIC, B.PERIODIC, B.OPEN)
        assert ei.value.code == B.EINVAL
        lo = torch.zeros(B.lbm_halo_elements(ctx), dtype=torch.float32, device="cuda")
        hi = torch.zeros_like(lo)
        with pytest.raises(B.LbmError) as ei:
            B.lbm_halo_pack(ctx, lo, hi)  # no step since the state was loaded
        assert ei.value.code == B.ESTATE
        with pytest.raises(B.LbmError) as ei:
            B.lbm_step(ctx, 2)
        assert ei.value.code == B.EINVAL
        B.lbm_step(ctx, 1)
        B.lbm_halo_pack(ctx, lo, hi)
        B.lbm_halo_unpack(ctx, hi, lo)
        assert B.lbm_check_finite(ctx)
        with pytest.raises(ValueError):
            B.lbm_halo_pack(ctx, lo[:-1], hi)
        # an open slab step admits no other call on the context until its end
        with pytest.raises(B.LbmError) as ei:
            B.lbm_slab_step_end(ctx, hi, lo)
        assert ei.value.code == B.ESTATE
        steps = B.lbm_step_count(ctx)
        B.lbm_slab_step_begin(ctx, lo, hi)
        for call in (lambda: B.lbm_slab_step_begin(ctx, lo, hi), lambda: B.lbm_step(ctx, 1),
                     lambda: B.lbm_halo_pack(ctx, lo, hi),
                     lambda: B.lbm_force_momentum_exchange(ctx),
                     lambda: B.lbm_set_body_force(ctx, 0.0, 0.0, 0.0)):
            with pytest.raises(B.LbmError) as ei:
                call()
            assert ei.value.code == B.ESTATE and "slab step" in str(ei.value)
        assert B.lbm_halo_elements(ctx) == 5 * 8 * 6 and B.lbm_step_count(ctx) == steps
        B.lbm_slab_step_end(ctx, hi, lo)
        assert B.lbm_step_count(ctx) == steps + 1
        assert B.lbm_check_finite(ctx)
        B.lbm_step(ctx, 1)
    finally:
        B.lbm_destroy(ctx)
