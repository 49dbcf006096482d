"""GPU (CUDA library through the C ABI) against the fp64 CPU oracle on identical seeded inputs.

Bar: max |f_gpu - f_oracle| <= 1e-5 on FLUID cells after N steps (fp32 storage and arithmetic
against fp64, rho ~ 1); bit-exact where the update is a pure permutation of integer labels."""
import math

import numpy as np
import pytest

import oracle
from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl
from lbm_harness import (LAYOUTS, SCHEMES, TOL_F, Case, max_fluid_diff, random_state, window)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def mixed_case(nx, ny, nz, faces, seed, solid=0.15, inlet_layer=True, g=(2e-5, -1e-5, 1e-5),
               tau=0.62, moving=0.0):
    """Random solids (a fraction `moving` of them moving walls), an optional inlet layer."""
    r = np.random.default_rng(seed)
    N = nx * ny * nz
    flags = (r.uniform(size=N) < solid).astype(np.uint8)
    if moving:
        flags[(flags == wl.SOLID) & (r.uniform(size=N) < moving)] = wl.MOVING_WALL
    if inlet_layer:
        x, _, _ = wl.coords(nx, ny, nz)
        flags[x == 0] = wl.INLET
    return Case(nx, ny, nz, tau, random_state(N, seed + 1), flags=flags, faces=faces,
                inlet=(1.01, 0.04, -0.01, 0.02), g=g, wall=(0.03, -0.02, 0.01))


# ---- small cases: every scheme x layout, all link types, ragged grids, even and odd counts -------

SMALL = [
    # nx, ny, nz, faces, solid fraction, inlet layer
    (37, 23, 19, (0, 0, 0), 0.0, False),
    (37, 23, 19, (0, 0, 0), 0.2, False),
    (33, 17, 9, (1, 0, 0), 0.15, True),
    (20, 19, 11, (1, 1, 0), 0.15, True),
    (13, 14, 15, (1, 1, 1), 0.1, False),
    (300, 3, 2, (1, 0, 1), 0.1, True),
]


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
@pytest.mark.parametrize("ci", range(len(SMALL)))
def test_small_cases_match_oracle(ci, layout, scheme):
    nx, ny, nz, faces, solid, inlet = SMALL[ci]
    case = mixed_case(nx, ny, nz, faces, 300 + ci, solid=solid, inlet_layer=inlet)
    for steps in (1, 4, 7):
        fo, Fo = case.run_oracle(steps, want_force=True)
        fg, Fg = case.run_gpu(steps, layout, scheme, want_force=True)
        assert max_fluid_diff(case, fg, fo) <= TOL_F, (steps, max_fluid_diff(case, fg, fo))
        scale = max(1.0, float(np.abs(Fo).max()))
        assert np.abs(Fg - Fo).max() <= 1e-4 * scale, (Fg, Fo)


MOVING = [
    # nx, ny, nz, faces, solid fraction, inlet layer
    (37, 23, 19, (0, 0, 0), 0.2, False),
    (33, 17, 9, (1, 0, 0), 0.15, True),
]


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
@pytest.mark.parametrize("ci", range(len(MOVING)))
def test_moving_walls_match_oracle(ci, layout, scheme):
    nx, ny, nz, faces, solid, inlet = MOVING[ci]
    case = mixed_case(nx, ny, nz, faces, 700 + ci, solid=solid, inlet_layer=inlet, moving=0.5)
    assert (case.flags == wl.MOVING_WALL).any()
    for steps in (1, 4, 7):
        fo, Fo = case.run_oracle(steps, want_force=True)
        fg, Fg = case.run_gpu(steps, layout, scheme, want_force=True)
        assert max_fluid_diff(case, fg, fo) <= TOL_F, (steps, max_fluid_diff(case, fg, fo))
        scale = max(1.0, float(np.abs(Fo).max()))
        assert np.abs(Fg - Fo).max() <= 1e-4 * scale, (Fg, Fo)


def test_couette_matches_oracle_and_is_linear():
    """Plane Couette flow (resting wall y = 0, lid y = ny - 1 moving at U along x), 16 x 18 x 16
    on the GPU against the oracle's 1 x 18 x 1 column (x/z invariance), 30000 steps."""
    ny, tau, U, steps = 18, 0.9, 0.02, 30000
    H = ny - 2
    def flags_for(nx, nz):
        _, y, _ = wl.coords(nx, ny, nz)
        fl = np.zeros(nx * ny * nz, np.uint8)
        fl[y == 0] = wl.SOLID
        fl[y == ny - 1] = wl.MOVING_WALL
        return fl
    col = Case(1, ny, 1, tau, oracle.equilibrium_field(*wl.uniform_fields(ny)),
               flags=flags_for(1, 1), wall=(U, 0, 0))
    fo, _ = col.run_oracle(steps)
    full = Case(16, ny, 16, tau, oracle.equilibrium_field(*wl.uniform_fields(16 * ny * 16)),
                flags=flags_for(16, 16), wall=(U, 0, 0))
    for scheme in ("AA", "AB"):
        fg, Fg = full.run_gpu(steps, "stream", scheme, want_force=True)
        fo_full = np.broadcast_to(fo.reshape(19, 1, ny, 1), (19, 16, ny, 16)).reshape(19, -1)
        assert max_fluid_diff(full, fg, fo_full) <= TOL_F
        F4 = fg.reshape(19, 16, ny, 16)
        with np.errstate(invalid="ignore"):  # wall cells hold 0
            ux = (F4 * oracle.tables()[0][:, 0, None, None, None]).sum(axis=0) / F4.sum(axis=0)
        y = np.arange(1, ny - 1)
        assert np.abs(ux[:, 1:ny - 1, :] - (U * (y - 0.5) / H)[None, :, None]).max() < 1e-3 * U
        # steady state: the shear forces on the two walls (rho nu U / H each, 16 x 16 cells)
        # cancel
        wall_force = (tau - 0.5) / 3 * U / H * 256
        assert abs(Fg[0]) < 1e-2 * wall_force


def test_lid_driven_cavity():
    """Lid-driven cavity: full parity at 32^3 (300 steps), AA == A-B, mass conservation."""
    n = 32
    flags = wl.cavity_flags(n, n, n)
    case = Case(n, n, n, 0.6, oracle.equilibrium_field(*wl.uniform_fields(n ** 3)), flags=flags,
                wall=(0.05, 0.0, 0.0))
    fo, Fo = case.run_oracle(300, want_force=True)
    fa, Fa = case.run_gpu(300, "stream", "AA", want_force=True)
    fb, Fb = case.run_gpu(300, "stream", "AB", want_force=True)
    assert max_fluid_diff(case, fa, fo) <= TOL_F
    assert max_fluid_diff(case, fb, fo) <= TOL_F
    assert np.abs(Fa - Fo).max() <= 1e-4 * max(1.0, np.abs(Fo).max())
    fl = case.fluid
    assert abs(fa[:, fl].sum() / case.f0_32[:, fl].astype(np.float64).sum() - 1) < 1e-6


@pytest.mark.slow
def test_lid_driven_cavity_256_windows_and_mass():
    n, k = 256, 3
    flags = wl.cavity_flags(n, n, n)
    r = np.random.default_rng(17).uniform(-1, 1, n ** 3).astype(np.float32)
    _, w, _ = oracle.tables()
    f0 = np.empty((19, n ** 3), np.float32)
    for q in range(19):
        f0[q] = np.float32(w[q]) * (1 + np.float32(0.01) * np.roll(r, 4099 * q))
    case = Case(n, n, n, 0.6, f0, flags=flags, wall=(0.05, 0.0, 0.0))
    fg, _ = case.run_gpu(k, "stream", "AA")
    # windows away from the non-periodic faces see exactly the full problem's cells
    for c in [(128, n - 2, 128), (1, n - 2, 1), (n - 2, 1, n - 2), (100, 200, 50), (5, 254, 250)]:
        sub, ci, _ = window(case, c, k + 1, f0)
        fo, _ = sub.run_oracle(k)
        nn = c[0] + n * (c[1] + n * c[2])
        assert np.abs(fg[:, nn] - fo[:, ci]).max() <= TOL_F, c
    ctx = case.gpu_context()
    try:
        m0 = case.f0_32[:, case.fluid].astype(np.float64).sum()
        B.lbm_step(ctx, 1000)
        f = np.zeros((19, case.N), np.float32)
        B.lbm_get_populations(ctx, f)
        assert B.lbm_check_finite(ctx)
    finally:
        B.lbm_destroy(ctx)
    assert abs(f[:, case.fluid].astype(np.float64).sum() / m0 - 1) < 1e-5


@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
def test_degenerate_grids(layout):
    """Grids of one cell, one row, one plane (a warp holding one or a few cells), in every layout;
    a thin 256 x 1 x 7 grid, whose tiled collision-layout pull has more blocks than the one-cell
    grid (its force partials are sized for both); and a two-cell row between an inlet and an open
    face."""
    for (nx, ny, nz) in [(1, 1, 1), (2, 1, 1), (1, 3, 1), (2, 2, 2), (5, 1, 7), (256, 1, 7)]:
        case = Case(nx, ny, nz, 0.7, random_state(nx * ny * nz, 7), g=(1e-4, 0, 0))
        fo, _ = case.run_oracle(5)
        for scheme in SCHEMES:
            fg, _ = case.run_gpu(5, layout, scheme)
            assert max_fluid_diff(case, fg, fo) <= TOL_F, ((nx, ny, nz), scheme)
    case = mixed_case(3, 2, 1, (1, 0, 0), 8, solid=0.0, inlet_layer=True)
    fo, _ = case.run_oracle(5)
    for scheme in SCHEMES:
        fg, _ = case.run_gpu(5, layout, scheme)
        assert max_fluid_diff(case, fg, fo) <= TOL_F, scheme


def test_zero_steps_is_identity_and_force_unavailable():
    case = mixed_case(9, 8, 7, (1, 0, 0), 5)
    ctx = case.gpu_context()
    try:
        B.lbm_step(ctx, 0)
        f = np.zeros((19, case.N), np.float32)
        B.lbm_get_populations(ctx, f)
        fl = case.fluid
        assert np.array_equal(f[:, fl], case.f0_32[:, fl])
        with pytest.raises(B.LbmError) as ei:
            B.lbm_force_momentum_exchange(ctx)
        assert ei.value.code == B.ESTATE
    finally:
        B.lbm_destroy(ctx)


@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_split_step_calls_equal_one_call(scheme):
    case = mixed_case(17, 9, 10, (1, 0, 0), 11)
    f1, F1 = case.run_gpu(9, "stream", scheme, want_force=True)
    f2, F2 = case.run_gpu(9, "stream", scheme, want_force=True, chunks=[2, 3, 1, 3])
    assert np.array_equal(f1, f2)
    assert np.array_equal(F1, F2)


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["bundle", "collision"])
@pytest.mark.parametrize("dims, faces", [((37, 6, 5), (1, 0, 0)), ((13, 9, 4), (0, 1, 1)),
                                         ((300, 3, 2), (1, 0, 1)), ((64, 5, 3), (0, 0, 0)),
                                         ((64, 9, 40), (0, 1, 0)), ((32, 16, 24), (1, 0, 1)),
                                         ((96, 11, 9), (1, 1, 1)), ((64, 21, 40), (0, 1, 0)),
                                         ((32, 34, 20), (1, 0, 1)), ((32, 12, 6), (0, 0, 1))])
def test_layouts_bit_identical_to_stream(dims, faces, layout, scheme):
    """The layouts differ only in where a population is stored: the same collision in the same
    order gives identical populations in the bundle and collision layouts (the collision layout's
    own-population steps stage each warp's records through shared memory) and in the stream
    layout, on rows longer than a block, shorter than a warp and with a partial last warp.  With
    32 | nx the collision layout's A-B pull runs in 2.5D tiles: several z chunks (64 x 9 x 40,
    32 x 16 x 24), ragged tile rows (ny not a multiple of the tile's 8 rows), open faces on each
    axis; with also ny >= 10 its AA odd step runs in the same tiles, updated in place (32 x 16 x
    24, 96 x 11 x 9, 64 x 21 x 40, 32 x 34 x 20, and 32 x 12 x 6 in one chunk whose halo planes
    wrap onto its own planes)."""
    nx, ny, nz = dims
    case = mixed_case(nx, ny, nz, faces, 1900 + nx, solid=0.15, inlet_layer=True, moving=0.3)
    for steps in (1, 2, 5):
        fs, Fs = case.run_gpu(steps, "stream", scheme, want_force=True, pairs=False)
        fl_, Fl = case.run_gpu(steps, layout, scheme, want_force=True)
        fl = case.fluid
        assert np.array_equal(fl_[:, fl], fs[:, fl]), (steps, np.abs(fl_[:, fl] - fs[:, fl]).max())
        assert np.abs(Fl - Fs).max() <= 1e-6 * max(1.0, float(np.abs(Fs).max())), (steps, Fl, Fs)


@pytest.mark.parametrize("scheme", ["AA", "AB"])
@pytest.mark.parametrize("walls", ["moving_only", "none_inlet", "none"])
@pytest.mark.parametrize("dims, faces", [((32, 16, 24), (1, 0, 1)), ((96, 11, 9), (1, 1, 1)),
                                         ((64, 21, 40), (0, 1, 0)), ((32, 34, 20), (1, 0, 1)),
                                         ((64, 20, 17), (0, 0, 0)), ((32, 12, 6), (0, 0, 1))])
def test_collision_tiles_without_solid_links(dims, faces, walls, scheme):
    """A grid without SOLID cells runs the collision layout's tiled kernels without the
    bounce-back path; the tiled AA odd step then writes back the elements whose writer (the cell
    x - c_q of element q of the record of x) lies in the block's tile and chunk.  Moving walls
    only (their neighbours are special cells, stepped by the boundary kernel after the tiled
    step), an inlet layer (producers) or neither; open faces, ragged tile rows, several z chunks
    and one (32 x 12 x 6), nx = 32 (a halo column is the grid's other edge column).  Bit-identical to the stream layout, and
    within the parity bar of the oracle."""
    nx, ny, nz = dims
    moving = walls == "moving_only"
    case = mixed_case(nx, ny, nz, faces, 2300 + nx + ny, solid=0.15 if moving else 0.0,
                      inlet_layer=walls != "none", moving=1.0 if moving else 0.0)
    assert not (case.flags == wl.SOLID).any()
    for steps in (1, 2, 5):
        fs, Fs = case.run_gpu(steps, "stream", scheme, want_force=True, pairs=False)
        fc, Fc = case.run_gpu(steps, "collision", scheme, want_force=True)
        fl = case.fluid
        assert np.array_equal(fc[:, fl], fs[:, fl]), (steps, np.abs(fc[:, fl] - fs[:, fl]).max())
        assert np.abs(Fc - Fs).max() <= 1e-6 * max(1.0, float(np.abs(Fs).max())), (steps, Fc, Fs)
    fo, Fo = case.run_oracle(5, want_force=True)
    assert max_fluid_diff(case, fc, fo) <= TOL_F, max_fluid_diff(case, fc, fo)
    assert np.abs(Fc - Fo).max() <= 1e-4 * max(1.0, float(np.abs(Fo).max())), (Fc, Fo)


# ---- streaming is an exact permutation ---------------------------------------------------------------

@pytest.mark.parametrize("dims, faces", [((21, 10, 7), (0, 0, 0)), ((64, 20, 17), (1, 0, 1))])
@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
def test_streaming_permutation_bit_exact(layout, scheme, dims, faces):
    """Collision off (tau = 1e30, g = 0), integer labels: every label must land exactly where the
    oracle (pinned to forward particle tracing) puts it -- neighbour indexing is bit-exact.  The
    second grid takes the collision layout's tiled A-B pull and AA odd step (z chunks, open x and z
    faces)."""
    nx, ny, nz = dims
    r = np.random.default_rng(41)
    flags = (r.uniform(size=nx * ny * nz) < 0.2).astype(np.uint8)
    case = Case(nx, ny, nz, 1e30, wl.labels(nx * ny * nz), flags=flags, faces=faces)
    for steps in (1, 2, 5):
        fo, _ = case.run_oracle(steps)
        fg, _ = case.run_gpu(steps, layout, scheme)
        fl = case.fluid
        assert np.array_equal(fg[:, fl], fo[:, fl]), steps


# ---- configuration 1: periodic 32^3 Taylor-Green, 100 steps -----------------------------------------

@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_taylor_green_32_full(scheme):
    rho, u = wl.taylor_green(32, 32, 32, 0.02, noise=1e-4, seed=wl.SEED_TG32)
    case = Case(32, 32, 32, 0.6, oracle.equilibrium_field(rho, u))
    fo, _ = case.run_oracle(100)
    fg, _ = case.run_gpu(100, "stream", scheme)
    d = max_fluid_diff(case, fg, fo)
    print(f"\nfull-length parity taylor_green_32 {scheme} stream: all cells, max|df| {d:.3e}")
    assert d <= TOL_F


# ---- configuration 2: 64^3 channel, Guo forcing, 20000 steps -------------------------------------------

def test_channel_64_full_against_reduced_oracle():
    """The channel is invariant along x and z, so the 64^3 oracle equals the 1 x 64 x 1 oracle
    broadcast (pinned bit-exactly on the CPU); the GPU runs the full 64^3 problem."""
    n, tau, g, steps = 64, 0.8, 1e-6, 20000
    f0 = oracle.equilibrium_field(*wl.uniform_fields(n))
    col = Case(1, n, 1, tau, f0, flags=wl.channel_flags(1, n, 1), g=(g, 0, 0))
    fo, Fo = col.run_oracle(steps, want_force=True)
    full = Case(n, n, n, tau, oracle.equilibrium_field(*wl.uniform_fields(n ** 3)),
                flags=wl.channel_flags(n, n, n), g=(g, 0, 0))
    fg, Fg = full.run_gpu(steps, "stream", "AA", want_force=True)
    fo_full = np.broadcast_to(fo.reshape(19, 1, n, 1), (19, n, n, n)).reshape(19, -1)
    d = max_fluid_diff(full, fg, fo_full)
    print(f"\nfull-length parity channel_64 AA stream: all cells, max|df| {d:.3e}, force x "
          f"{Fg[0]:.6e} vs oracle {Fo[0] * n * n:.6e}")
    assert d <= TOL_F
    assert abs(Fg[0] - Fo[0] * n * n) <= 1e-3 * abs(Fo[0] * n * n)
    # the profile: parabola with the startup transient (same bar as the oracle's own pin)
    ctx = full.gpu_context()
    try:
        B.lbm_step(ctx, steps)
        rho = np.zeros(full.N, np.float32)
        u = np.zeros(3 * full.N, np.float32)
        B.lbm_macroscopic(ctx, rho, u)
    finally:
        B.lbm_destroy(ctx)
    ux = u[:full.N].reshape(n, n, n)[:, 1:n - 1, :].mean(axis=(0, 2))
    nu, H = (tau - 0.5) / 3, n - 2
    eta = np.arange(1, n - 1) - 0.5
    expect = g / (2 * nu) * eta * (H - eta)
    for m in range(1, 400, 2):
        expect -= (4 * g * H * H / (nu * math.pi ** 3 * m ** 3)) * np.sin(m * math.pi * eta / H) \
            * math.exp(-m * m * math.pi ** 2 * nu * steps / (H * H))
    assert np.abs(ux - expect).max() < 0.01 * g * H * H / (8 * nu)


# ---- configuration 3: periodic 128^3 Taylor-Green, AA vs A-B across layouts -----------------------

def test_taylor_green_128_layouts_and_schemes():
    rho, u = wl.taylor_green(128, 128, 128, 0.05)
    case = Case(128, 128, 128, 0.6, oracle.equilibrium_field(rho, u))
    steps = 20
    fo, _ = case.run_oracle(steps)
    ref = None
    for layout in LAYOUTS:
        for scheme in ("AA", "AB"):
            fg, _ = case.run_gpu(steps, layout, scheme)
            assert max_fluid_diff(case, fg, fo) <= TOL_F, (layout, scheme)
            if ref is None:
                ref = fg
            else:
                assert np.abs(fg - ref).max() <= 1e-6, (layout, scheme)


# ---- configuration 4: sphere with inlet and open outlet ---------------------------------------------

def sphere_case(nx, ny, nz, center, r, tau=0.56, u_in=0.05):
    flags = wl.sphere_flags(nx, ny, nz, center, r)
    f0 = oracle.equilibrium_field(*wl.uniform_fields(nx * ny * nz, 1.0, (u_in, 0, 0)))
    return Case(nx, ny, nz, tau, f0, flags=flags, faces=(1, 0, 0), inlet=(1.0, u_in, 0.0, 0.0))


@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_sphere_reduced_full_run(scheme):
    case = sphere_case(48, 32, 32, (15, 16, 16), 5)
    fo, Fo = case.run_oracle(300, want_force=True)
    fg, Fg = case.run_gpu(300, "stream", scheme, want_force=True)
    assert max_fluid_diff(case, fg, fo) <= TOL_F
    assert np.abs(Fg - Fo).max() <= 1e-4 * abs(Fo[0])
    assert Fg[0] > 0


def test_sphere_128_windows_and_symmetry():
    case = sphere_case(128, 128, 128, (40, 64, 64), 16)
    k = 3
    fg, _ = case.run_gpu(k, "stream", "AA")
    centers = [(40, 64, 48 - 1), (24, 64, 64), (56, 70, 64), (100, 5, 120), (64, 64, 81)]
    for c in centers:
        sub, ci, _ = window(case, c, k + 1, case.f0_32)
        fo, _ = sub.run_oracle(k)
        if sub.flags[ci] != wl.FLUID:
            continue
        n = c[0] + 128 * (c[1] + 128 * c[2])
        assert np.abs(fg[:, n] - fo[:, ci]).max() <= TOL_F, c
    # full run: the drag is along +x, the transverse force vanishes by mirror symmetry
    ctx = case.gpu_context()
    try:
        B.lbm_step(ctx, 2000)
        F = B.lbm_force_momentum_exchange(ctx)
        assert B.lbm_check_finite(ctx)
    finally:
        B.lbm_destroy(ctx)
    assert F[0] > 0
    assert abs(F[1]) <= 1e-4 * F[0] and abs(F[2]) <= 1e-4 * F[0]


# ---- configuration 5: porous medium with body force ----------------------------------------------------

@pytest.mark.parametrize("scheme", ["AA", "AB"])
def test_porous_reduced_full_run(scheme):
    n = 48
    flags = wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512)
    case = Case(n, n, n, 0.7, random_state(n ** 3, 77, amp=5e-3, du=0.02), flags=flags,
                g=(1e-4, 0, 0))
    fo, Fo = case.run_oracle(60, want_force=True)
    fg, Fg = case.run_gpu(60, "stream", scheme, want_force=True)
    assert max_fluid_diff(case, fg, fo) <= TOL_F
    assert np.abs(Fg - Fo).max() <= 1e-4 * np.abs(Fo).max()


@pytest.mark.slow
def test_porous_512_windows():
    """Full 512^3 porous problem in the benchmark's configuration (AA, stream layout), checked on
    sampled cells against the oracle on their light cones; a random initial state makes every
    link carry a distinct value."""
    n = 512
    flags = wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512)
    N = n ** 3
    # near-equilibrium random state: one random field, shifted differently per population
    r = np.random.default_rng(5).uniform(-1, 1, N).astype(np.float32)
    _, w, _ = oracle.tables()
    f0 = np.empty((19, N), np.float32)
    for q in range(19):
        f0[q] = np.float32(w[q]) * (1 + np.float32(0.01) * np.roll(r, 7919 * q))
    case = Case(n, n, n, 0.7, f0, flags=flags, g=(1e-6, 0, 0))
    k = 4
    fg, _ = case.run_gpu(k, "stream", "AA")
    rs = np.random.default_rng(9)
    centers = [tuple(int(v) for v in rs.integers(0, n, 3)) for _ in range(12)]
    centers += [(0, 0, 0), (511, 511, 511), (0, 255, 511)]
    checked = 0
    for c in centers:
        sub, ci, _ = window(case, c, k + 1, f0)
        if sub.flags[ci] != wl.FLUID:
            continue
        fo, _ = sub.run_oracle(k)
        nn = c[0] + n * (c[1] + n * c[2])
        assert np.abs(fg[:, nn] - fo[:, ci]).max() <= TOL_F, c
        checked += 1
    assert checked >= 5


# ---- state handling ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["stream", "bundle", "collision"])
def test_macroscopic_and_host_paths(layout):
    case = mixed_case(19, 13, 11, (1, 0, 0), 21)
    P = case.oracle_problem()
    for steps in (0, 3, 4):
        fo, _ = P.step_ab(case.f0_32.astype(np.float64), steps)
        ro, uo = P.macroscopic(fo)
        for device_input in (True, False):
            ctx = case.gpu_context(layout, "AA", device_input=device_input)
            try:
                B.lbm_step(ctx, steps)
                rho = np.zeros(case.N, np.float32)
                u = np.zeros(3 * case.N, np.float32)
                B.lbm_macroscopic(ctx, rho, u)
                rho_d = torch.zeros(case.N, dtype=torch.float32, device="cuda")
                u_d = torch.zeros(3 * case.N, dtype=torch.float32, device="cuda")
                B.lbm_macroscopic(ctx, rho_d, u_d)
                f_d = torch.zeros(19 * case.N, dtype=torch.float32, device="cuda")
                B.lbm_get_populations(ctx, f_d)
            finally:
                B.lbm_destroy(ctx)
            assert np.array_equal(rho, rho_d.cpu().numpy())
            assert np.array_equal(u, u_d.cpu().numpy())
            assert np.abs(rho - ro).max() <= 1e-5
            assert np.abs(u.reshape(3, -1) - uo).max() <= 1e-5
            fl = case.fluid
            assert np.abs(f_d.cpu().numpy().reshape(19, -1)[:, fl] - fo[:, fl]).max() <= TOL_F


def test_set_equilibrium_matches_oracle():
    n = 24
    rho, u = wl.taylor_green(n, n, n, 0.05, noise=1e-3, seed=3)
    feq = oracle.equilibrium_field(rho, u)
    ctx = B.lbm_create(n, n, n, 0.6)
    try:
        B.lbm_set_equilibrium(ctx, rho.astype(np.float32), u.astype(np.float32).reshape(-1))
        f = np.zeros((19, n ** 3), np.float32)
        B.lbm_get_populations(ctx, f)
    finally:
        B.lbm_destroy(ctx)
    assert np.abs(f - feq).max() <= 1e-6


def test_invalid_flags_leave_state_unchanged():
    case = mixed_case(9, 8, 7, (0, 0, 0), 31, inlet_layer=False)
    ctx = case.gpu_context()
    try:
        bad = case.flags.copy()
        bad[17] = 7
        with pytest.raises(B.LbmError) as ei:
            B.lbm_set_flags(ctx, bad)
        assert ei.value.code == B.EINVAL
        B.lbm_step(ctx, 3)
        f = np.zeros((19, case.N), np.float32)
        B.lbm_get_populations(ctx, f)
    finally:
        B.lbm_destroy(ctx)
    fo, _ = case.run_oracle(3)
    assert max_fluid_diff(case, f.astype(np.float64), fo) <= TOL_F


def test_check_finite_flags_nan():
    case = mixed_case(8, 8, 8, (0, 0, 0), 33, solid=0.0, inlet_layer=False)
    f0 = case.f0_32.copy()
    f0[5, 100] = np.nan
    ctx = B.lbm_create(8, 8, 8, 0.7)
    try:
        B.lbm_set_populations(ctx, case.f0_32)
        assert B.lbm_check_finite(ctx)
        B.lbm_set_populations(ctx, f0)
        assert not B.lbm_check_finite(ctx)
    finally:
        B.lbm_destroy(ctx)


def test_stream_profile_and_launch_counts():
    case = mixed_case(16, 16, 16, (1, 0, 0), 35)
    ctx = case.gpu_context()
    try:
        s = torch.cuda.Stream()
        B.lbm_set_stream(ctx, s.cuda_stream)
        B.lbm_profile_enable(ctx, True)
        before = B.lbm_kernel_launches(ctx)
        B.lbm_step(ctx, 4)
        s.synchronize()
        launched = B.lbm_kernel_launches(ctx) - before
        # 2 even + 2 odd + 2 boundary-cell odd + 2 open-face pre-gathers (both x faces in one
        # launch) + 2 force-sum stages
        assert launched == 2 + 2 + 2 + 2 + 2
        n_even, ms_even = B.lbm_profile_read(ctx, B.K_AA_EVEN)
        n_odd, ms_odd = B.lbm_profile_read(ctx, B.K_AA_ODD)
        assert n_even == 2 and n_odd == 2 and ms_even > 0 and ms_odd > 0
        assert B.lbm_step_count(ctx) == 4
    finally:
        B.lbm_destroy(ctx)


# ---- full-length runs: properties that hold at any size ------------------------------------------

def gpu_moments(ctx, N, g):
    """(mass, momentum[3]) of the natural state from lbm_macroscopic, summed in fp64:
    j = rho (u - g/2) undoes the reported half-force shift."""
    rho = torch.zeros(N, dtype=torch.float32, device="cuda")
    u = torch.zeros(3 * N, dtype=torch.float32, device="cuda")
    B.lbm_macroscopic(ctx, rho, u)
    r = rho.double()
    u = u.double().view(3, N)
    j = [(r * (u[a] - 0.5 * g[a])).sum().item() for a in range(3)]
    return r.sum().item(), np.array(j)


@pytest.mark.slow
def test_taylor_green_128_full_length_properties():
    """1000 steps at 128^3: every scheme and layout agrees, mass and momentum are conserved."""
    n = 128
    rho, u = wl.taylor_green(n, n, n, 0.05)
    case = Case(n, n, n, 0.6, oracle.equilibrium_field(rho, u))
    ref = None
    for layout in LAYOUTS:
        for scheme in ("AA", "AB"):
            ctx = case.gpu_context(layout, scheme)
            try:
                m0, j0 = gpu_moments(ctx, case.N, (0, 0, 0))
                B.lbm_step(ctx, 1000)
                m1, j1 = gpu_moments(ctx, case.N, (0, 0, 0))
                f = torch.zeros(19 * case.N, dtype=torch.float32, device="cuda")
                B.lbm_get_populations(ctx, f)
            finally:
                B.lbm_destroy(ctx)
            assert abs(m1 / m0 - 1) < 1e-6
            assert np.abs(j1 - j0).max() < 1e-6 * m0
            if ref is None:
                ref = f
            else:
                assert (f - ref).abs().max().item() <= 1e-6, (layout, scheme)


@pytest.mark.slow
def test_sphere_128_full_length_aa_equals_ab():
    case = sphere_case(128, 128, 128, (40, 64, 64), 16)
    fa, Fa = case.run_gpu(2000, "stream", "AA", want_force=True)
    fb, Fb = case.run_gpu(2000, "stream", "AB", want_force=True)
    assert max_fluid_diff(case, fa, fb) <= 1e-6
    assert np.abs(Fa - Fb).max() <= 1e-5 * abs(Fa[0])


@pytest.mark.slow
def test_porous_512_conservation_and_momentum_balance():
    """The benchmark configuration (porous 512^3, AA, stream layout, Guo g = 1e-6, tau 0.7):
    bounce-back conserves mass exactly, and over every step the fluid momentum grows by the body
    force minus the momentum handed to the solids (the momentum-exchange force of that step)."""
    n, g = 512, (1e-6, 0.0, 0.0)
    N = n ** 3
    flags = wl.porous_flags(n, n, n, 0.30, 3, seed=wl.SEED_POROUS512)
    ctx = B.lbm_create(n, n, n, 0.7, B.LAYOUT_STREAM, B.STREAMING_AA)
    try:
        B.lbm_set_flags(ctx, flags)
        B.lbm_set_body_force(ctx, *g)
        rho = torch.ones(N, dtype=torch.float32, device="cuda")
        u = torch.zeros(3 * N, dtype=torch.float32, device="cuda")
        B.lbm_set_equilibrium(ctx, rho, u)
        B.lbm_step(ctx, 20)
        m_prev, j_prev = gpu_moments(ctx, N, g)
        for _ in range(3):
            B.lbm_step(ctx, 1)
            F = B.lbm_force_momentum_exchange(ctx)
            m, j = gpu_moments(ctx, N, g)
            body = m_prev * g[0]
            assert abs(m / m_prev - 1) < 1e-6
            assert abs((j[0] - j_prev[0]) - (body - F[0])) <= 1e-3 * body
            assert abs((j[1] - j_prev[1]) + F[1]) <= 1e-3 * body
            assert abs((j[2] - j_prev[2]) + F[2]) <= 1e-3 * body
            m_prev, j_prev = m, j
        assert B.lbm_check_finite(ctx)
    finally:
        B.lbm_destroy(ctx)


# ---- graph replay --------------------------------------------------------------------------------

@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
def test_graph_replay_equals_direct_launches(scheme):
    """lbm_step replays captured CUDA graphs in chunks; the result must equal one-by-one
    launches bit for bit, for step counts below, at and across the chunk length, and across
    a change of body force (which drops the cached graphs)."""
    case = mixed_case(23, 12, 9, (1, 0, 0), 61)
    out = []
    for graphs in (True, False):
        ctx = case.gpu_context("stream", scheme)
        try:
            B.lbm_set_graph_launch(ctx, graphs)
            res = []
            for n in (1, 2, 5, 32, 33, 70):
                B.lbm_step(ctx, n)
                res.append(B.lbm_force_momentum_exchange(ctx))
            B.lbm_set_body_force(ctx, -3e-5, 1e-5, 0.0)
            B.lbm_step(ctx, 9)
            res.append(B.lbm_force_momentum_exchange(ctx))
            f = np.zeros((19, case.N), np.float32)
            B.lbm_get_populations(ctx, f)
            assert B.lbm_step_count(ctx) == 1 + 2 + 5 + 32 + 33 + 70 + 9
        finally:
            B.lbm_destroy(ctx)
        out.append((f, res))
    assert np.array_equal(out[0][0], out[1][0])
    for a, b in zip(out[0][1], out[1][1]):
        assert np.array_equal(a, b)


# ---- half-precision storage (LBM_LAYOUT_STREAM_FP16) ---------------------------------------------

from lbm_harness import fp16_tolerance  # noqa: E402


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("ci", range(len(SMALL)))
def test_fp16_storage_equals_fp32_within_rounding(ci, scheme):
    """Same kernels, populations stored in half precision: equal to the fp32 layout within the
    fp16 rounding bound (an indexing error would show as O(1e-2) differences)."""
    nx, ny, nz, faces, solid, inlet = SMALL[ci]
    case = mixed_case(nx, ny, nz, faces, 300 + ci, solid=solid, inlet_layer=inlet)
    for steps in (1, 4, 7):
        f32, F32 = case.run_gpu(steps, "stream", scheme, want_force=True)
        f16, F16 = case.run_gpu(steps, "stream_fp16", scheme, want_force=True)
        tol = fp16_tolerance(case.f0_32, steps)
        assert max_fluid_diff(case, f16, f32) <= tol, (steps, max_fluid_diff(case, f16, f32), tol)


def test_fp16_taylor_green_against_oracle():
    rho, u = wl.taylor_green(32, 32, 32, 0.02, noise=1e-4, seed=wl.SEED_TG32)
    case = Case(32, 32, 32, 0.6, oracle.equilibrium_field(rho, u))
    fo, _ = case.run_oracle(100)
    for scheme in ("AA", "AB"):
        fg, _ = case.run_gpu(100, "stream_fp16", scheme)
        assert max_fluid_diff(case, fg, fo) <= fp16_tolerance(case.f0_32, 100)


# ---- two-cell kernels (lbm_set_cell_pairs) ---------------------------------------------------------

PAIR_CASES = [
    # nx even; nx, ny, nz, faces, solid fraction, inlet layer, moving fraction of the solids
    (38, 23, 19, (0, 0, 0), 0.0, False, 0.0),
    (38, 23, 19, (0, 0, 0), 0.25, False, 0.0),
    (34, 17, 9, (1, 0, 0), 0.15, True, 0.0),
    (20, 19, 11, (1, 1, 0), 0.15, True, 0.3),
    (14, 14, 15, (1, 1, 1), 0.1, False, 0.0),
    (16, 12, 10, (0, 0, 0), 0.2, False, 0.5),
    (2, 5, 3, (0, 0, 0), 0.2, False, 0.0),
    (4, 3, 2, (1, 0, 0), 0.1, True, 0.0),
    (300, 3, 2, (1, 0, 1), 0.1, True, 0.0),
]


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["stream", "stream_fp16", "bundle"])
@pytest.mark.parametrize("ci", range(len(PAIR_CASES)))
def test_cell_pairs_bit_identical_to_one_cell_kernels(ci, layout, scheme):
    """The two-cell kernels do the same arithmetic in the same order as the one-cell kernels:
    identical populations after every number of steps; the force (partial sums grouped per
    thread) within 1e-5 relative.  In the bundle layout every step but AB2's streaming pass has a
    two-cell kernel."""
    nx, ny, nz, faces, solid, inlet, moving = PAIR_CASES[ci]
    case = mixed_case(nx, ny, nz, faces, 700 + ci, solid=solid, inlet_layer=inlet, moving=moving)
    for steps in (1, 2, 5):
        f2, F2 = case.run_gpu(steps, layout, scheme, want_force=True, pairs=True)
        f1, F1 = case.run_gpu(steps, layout, scheme, want_force=True, pairs=False)
        fl = case.fluid
        assert np.array_equal(f2[:, fl], f1[:, fl]), (steps, np.abs(f2[:, fl] - f1[:, fl]).max())
        scale = max(1.0, float(np.abs(F1).max()))
        assert np.abs(F2 - F1).max() <= 1e-5 * scale, (steps, F2, F1)


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("ci", range(len(PAIR_CASES)))
def test_cell_pairs_match_oracle(ci, scheme):
    nx, ny, nz, faces, solid, inlet, moving = PAIR_CASES[ci]
    case = mixed_case(nx, ny, nz, faces, 800 + ci, solid=solid, inlet_layer=inlet, moving=moving)
    fo, Fo = case.run_oracle(7, want_force=True)
    for layout in (("stream", "bundle") if scheme == "AA" else ("stream",)):
        fg, Fg = case.run_gpu(7, layout, scheme, want_force=True, pairs=True)
        assert max_fluid_diff(case, fg, fo) <= TOL_F, layout
        assert np.abs(Fg - Fo).max() <= 1e-4 * max(1.0, float(np.abs(Fo).max())), layout


# ---- boundary kernel beside the main kernel (lbm_set_boundary_overlap) ------------------------------

# cases with special cells (inlet layers, open faces, moving walls); the last one large enough
# that the boundary and main kernels run at the same time on the device
OVERLAP_CASES = [2, 3, 4, 5, 7, 8, (96, 48, 40, (1, 0, 0), 0.1, True, 0.2)]


@pytest.mark.parametrize("graphs", [True, False])
@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("layout", ["stream", "stream_fp16", "bundle", "collision"])
@pytest.mark.parametrize("ci", range(len(OVERLAP_CASES)))
def test_boundary_overlap_bit_identical(ci, layout, scheme, pairs, graphs):
    """The boundary kernel on its own stream beside the main kernel stores into slots the main
    kernel leaves alone: populations and force are identical to the serial order."""
    spec = OVERLAP_CASES[ci]
    nx, ny, nz, faces, solid, inlet, moving = PAIR_CASES[spec] if isinstance(spec, int) else spec
    case = mixed_case(nx, ny, nz, faces, 960 + ci, solid=solid, inlet_layer=inlet, moving=moving)
    for steps in (3, 6):
        fo, Fo = case.run_gpu(steps, layout, scheme, want_force=True, pairs=pairs, graphs=graphs,
                              overlap=True)
        fs, Fs = case.run_gpu(steps, layout, scheme, want_force=True, pairs=pairs, graphs=graphs,
                              overlap=False)
        fl = case.fluid
        assert np.array_equal(fo[:, fl], fs[:, fl]), (steps, np.abs(fo[:, fl] - fs[:, fl]).max())
        assert np.array_equal(Fo, Fs), (steps, Fo, Fs)


def test_boundary_overlap_large_case_matches_oracle():
    """The overlapped AA and A-B steps on the large overlap case against the oracle."""
    nx, ny, nz, faces, solid, inlet, moving = OVERLAP_CASES[-1]
    case = mixed_case(nx, ny, nz, faces, 990, solid=solid, inlet_layer=inlet, moving=moving)
    fo, Fo = case.run_oracle(6, want_force=True)
    for scheme in ("AA", "AB"):
        fg, Fg = case.run_gpu(6, "stream", scheme, want_force=True)
        assert max_fluid_diff(case, fg, fo) <= TOL_F, scheme
        assert np.abs(Fg - Fo).max() <= 1e-4 * max(1.0, float(np.abs(Fo).max())), scheme


def test_cell_pairs_eligibility():
    def state(nx, layout, allow=True):
        ctx = B.lbm_create(nx, 6, 4, 0.6, layout, B.STREAMING_AA)
        try:
            return B.lbm_set_cell_pairs(ctx, allow)
        finally:
            B.lbm_destroy(ctx)
    assert state(8, B.LAYOUT_STREAM) is True
    assert state(8, B.LAYOUT_STREAM_FP16) is True
    assert state(8, B.LAYOUT_STREAM, allow=False) is False
    assert state(7, B.LAYOUT_STREAM) is False
    assert state(8, B.LAYOUT_BUNDLE) is False
    assert state(8, B.LAYOUT_COLLISION) is False


def test_cell_pairs_with_graphs_and_chunks():
    """Toggling the kernel family between lbm_step calls (graphs dropped and recaptured) and
    splitting the steps leaves the result unchanged."""
    case = mixed_case(24, 10, 8, (0, 0, 0), 901, solid=0.2, inlet_layer=False, moving=0.3)
    ref, _ = case.run_gpu(40, "stream", "AA", pairs=False)
    ctx = case.gpu_context("stream", "AA")
    try:
        for i, n in enumerate((3, 32, 5)):
            B.lbm_set_cell_pairs(ctx, i != 1)
            B.lbm_step(ctx, n)
        f = np.zeros((19, case.N), np.float32)
        B.lbm_get_populations(ctx, f)
    finally:
        B.lbm_destroy(ctx)
    assert np.array_equal(f.astype(np.float64)[:, case.fluid], ref[:, case.fluid])


@pytest.mark.parametrize("graphs", [True, False])
@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("geometry", ["periodic", "inlet_open_x"])
def test_flags_changed_between_even_and_odd_step(geometry, pairs, graphs):
    """AA: new SOLID cells set after an even step.  The odd step that follows bounces back from
    them (the two-cell kernels first write the pre-bounced values the new flags need); the result
    matches the oracle run the same way, flags1 for one step, flags2 after."""
    nx, ny, nz, tau, g = 20, 14, 12, 0.63, (1e-5, -2e-5, 0.0)
    N = nx * ny * nz
    r = np.random.default_rng(950)
    flags1 = (r.uniform(size=N) < 0.15).astype(np.uint8)
    faces = (0, 0, 0)
    if geometry == "inlet_open_x":
        x, _, _ = wl.coords(nx, ny, nz)
        flags1[x == 0] = wl.INLET
        faces = (1, 0, 0)
    flags2 = flags1.copy()
    flags2[(flags1 == wl.FLUID) & (r.uniform(size=N) < 0.1)] = wl.SOLID
    inlet = (1.01, 0.03, 0.0, 0.0)
    f0 = random_state(N, 951)
    P1 = oracle.Problem(nx, ny, nz, tau, flags=flags1, faces=faces, inlet=inlet, g=g)
    P2 = oracle.Problem(nx, ny, nz, tau, flags=flags2, faces=faces, inlet=inlet, g=g)
    A, _ = P1.step_aa(f0, 0, 1)
    A, _ = P2.step_aa(A, 1, 5)          # steps 2..6: natural state after an even count
    case = Case(nx, ny, nz, tau, f0, flags=flags1, faces=faces, inlet=inlet, g=g)
    ctx = case.gpu_context("stream", "AA", pairs=pairs)
    try:
        B.lbm_set_graph_launch(ctx, graphs)
        B.lbm_step(ctx, 1)
        B.lbm_set_flags(ctx, flags2)
        B.lbm_step(ctx, 1)
        B.lbm_step(ctx, 4)
        f = np.zeros((19, N), np.float32)
        B.lbm_get_populations(ctx, f)
    finally:
        B.lbm_destroy(ctx)
    fl = flags2 == wl.FLUID
    assert np.abs(f.astype(np.float64)[:, fl] - A[:, fl]).max() <= TOL_F


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("k", [1, 2])
@pytest.mark.parametrize("change", ["inlet_state", "new_inlet_cells"])
def test_inlet_change_between_steps(change, k, scheme, pairs):
    """INLET cells are producers: their post-collision slots carry f_eq(rho_in, u_in) for the next
    step's pulls.  A change of the inlet state, or FLUID cells turned INLET, after k steps acts on
    the streaming still pending: in a post-collision state (AA after an odd k, AB after any k) the
    last step's streaming happens under the new problem.  The collision of a cell that stays FLUID
    does not depend on the flags or the inlet, so the oracle reference is the old problem for k - 1
    steps and the new one for the rest (k and the rest when no streaming is pending)."""
    nx, ny, nz, tau, g = 18, 12, 10, 0.64, (1e-5, 0.0, -1e-5)
    N = nx * ny * nz
    r = np.random.default_rng(960 + k)
    x, _, _ = wl.coords(nx, ny, nz)
    flags1 = (r.uniform(size=N) < 0.1).astype(np.uint8)
    flags1[x == 0] = wl.INLET
    faces = (1, 0, 0)
    inlet1 = (1.01, 0.03, 0.0, 0.0)
    flags2, inlet2 = flags1.copy(), inlet1
    if change == "inlet_state":
        inlet2 = (0.99, 0.05, 0.01, -0.01)
    else:
        flags2[(flags1 == wl.FLUID) & (r.uniform(size=N) < 0.05)] = wl.INLET
    f0 = random_state(N, 961)
    P1 = oracle.Problem(nx, ny, nz, tau, flags=flags1, faces=faces, inlet=inlet1, g=g)
    P2 = oracle.Problem(nx, ny, nz, tau, flags=flags2, faces=faces, inlet=inlet2, g=g)
    pending = scheme == "AB" or (scheme == "AA" and k % 2 == 1)
    k1 = k - 1 if pending else k
    fo, _ = P1.step_ab(f0, k1)
    fo, _ = P2.step_ab(fo, k + 5 - k1)
    case = Case(nx, ny, nz, tau, f0, flags=flags1, faces=faces, inlet=inlet1, g=g)
    ctx = case.gpu_context("stream", scheme, pairs=pairs)
    try:
        B.lbm_step(ctx, k)
        if change == "inlet_state":
            B.lbm_set_inlet(ctx, *inlet2)
        else:
            B.lbm_set_flags(ctx, flags2)
        B.lbm_step(ctx, 5)
        f = np.zeros((19, N), np.float32)
        B.lbm_get_populations(ctx, f)
    finally:
        B.lbm_destroy(ctx)
    fl = flags2 == wl.FLUID
    assert np.abs(f.astype(np.float64)[:, fl] - fo[:, fl]).max() <= TOL_F


# ---- TMA-staged AA odd step (lbm_set_tma_gather) --------------------------------------------------

TMA_CASES = [
    # 16 | nx <= 512; nx, ny, nz, faces, solid fraction, inlet layer, moving fraction
    (32, 23, 19, (0, 0, 0), 0.0, False, 0.0),
    (32, 23, 19, (0, 0, 0), 0.25, False, 0.0),
    (48, 17, 9, (1, 0, 0), 0.15, True, 0.0),
    (16, 19, 11, (1, 1, 0), 0.15, True, 0.3),
    (64, 14, 15, (1, 1, 1), 0.1, False, 0.0),
    (16, 12, 10, (0, 0, 0), 0.2, False, 0.5),
    (16, 1, 1, (0, 0, 0), 0.0, False, 0.0),
    (512, 3, 2, (1, 0, 1), 0.1, True, 0.0),
    (96, 33, 5, (0, 1, 0), 0.3, False, 0.2),
]


@pytest.mark.parametrize("layout", ["stream", "stream_fp16"])
@pytest.mark.parametrize("ci", range(len(TMA_CASES)))
def test_tma_gather_bit_identical(ci, layout):
    """The staged odd step reads the same slots as the register one: identical populations after
    odd and even step counts; the force within 1e-5 relative (its partial sums are grouped by the
    persistent CTAs)."""
    nx, ny, nz, faces, solid, inlet, moving = TMA_CASES[ci]
    case = mixed_case(nx, ny, nz, faces, 1100 + ci, solid=solid, inlet_layer=inlet, moving=moving)
    for steps in (2, 5, 8):
        f1, F1 = case.run_gpu(steps, layout, "AA", want_force=True, tma=True)
        f0, F0 = case.run_gpu(steps, layout, "AA", want_force=True, tma=False)
        fl = case.fluid
        assert np.array_equal(f1[:, fl], f0[:, fl]), (steps, np.abs(f1[:, fl] - f0[:, fl]).max())
        scale = max(1.0, float(np.abs(F0).max()))
        assert np.abs(F1 - F0).max() <= 1e-5 * scale, (steps, F1, F0)


@pytest.mark.parametrize("ci", [1, 3, 8])
def test_tma_gather_matches_oracle(ci):
    nx, ny, nz, faces, solid, inlet, moving = TMA_CASES[ci]
    case = mixed_case(nx, ny, nz, faces, 1200 + ci, solid=solid, inlet_layer=inlet, moving=moving)
    fo, Fo = case.run_oracle(9, want_force=True)
    fg, Fg = case.run_gpu(9, "stream", "AA", want_force=True, tma=True)
    assert max_fluid_diff(case, fg, fo) <= TOL_F
    assert np.abs(Fg - Fo).max() <= 1e-4 * max(1.0, float(np.abs(Fo).max()))


def test_tma_gather_eligibility():
    def state(nx, layout=B.LAYOUT_STREAM, pairs=True, allow=True):
        ctx = B.lbm_create(nx, 6, 4, 0.6, layout, B.STREAMING_AA)
        try:
            B.lbm_set_cell_pairs(ctx, pairs)
            return B.lbm_set_tma_gather(ctx, allow)
        finally:
            B.lbm_destroy(ctx)
    assert state(16) is True
    assert state(512) is True
    assert state(32, B.LAYOUT_STREAM_FP16) is True
    assert state(32, allow=False) is False
    assert state(32, pairs=False) is False
    assert state(20) is False
    assert state(8) is False
    assert state(528) is False
    assert state(32, B.LAYOUT_BUNDLE) is False


def test_tma_gather_with_graphs_and_toggles():
    case = mixed_case(64, 10, 8, (0, 0, 0), 1301, solid=0.2, inlet_layer=False, moving=0.3)
    ref, _ = case.run_gpu(41, "stream", "AA", tma=False)
    ctx = case.gpu_context("stream", "AA")
    try:
        for i, n in enumerate((3, 32, 6)):
            B.lbm_set_tma_gather(ctx, i != 1)
            B.lbm_step(ctx, n)
        f = np.zeros((19, case.N), np.float32)
        B.lbm_get_populations(ctx, f)
        assert B.lbm_check_finite(ctx)
    finally:
        B.lbm_destroy(ctx)
    assert np.array_equal(f.astype(np.float64)[:, case.fluid], ref[:, case.fluid])


def test_tma_gather_wait_timeout_is_reported(monkeypatch):
    """Failure detection without a GPU fault: with the test hook the staged odd step announces 16
    bytes more than it copies, so its wait can never complete.  The wait gives up after its 2 s
    bound, the kernel drains its own copies and returns, and the next synchronising call reports
    LBM_ETIMEOUT.  The device stays usable."""
    import time
    monkeypatch.setenv("LBM_TEST_STAGE_TIMEOUT", "1")
    case = Case(32, 4, 2, 0.7, random_state(32 * 4 * 2, 1500))
    ctx = case.gpu_context("stream", "AA", tma=True)
    try:
        assert B.lbm_set_tma_gather(ctx, True)
        B.lbm_set_graph_launch(ctx, False)
        t0 = time.time()
        B.lbm_step(ctx, 2)
        f = np.zeros((19, case.N), np.float32)
        with pytest.raises(B.LbmError) as ei:
            B.lbm_get_populations(ctx, f)
        assert ei.value.code == B.ETIMEOUT
        assert "gave up waiting" in str(ei.value)
        assert time.time() - t0 < 60
    finally:
        B.lbm_destroy(ctx)
    monkeypatch.delenv("LBM_TEST_STAGE_TIMEOUT")
    fg, _ = case.run_gpu(2, "stream", "AA", tma=True)
    fo, _ = case.run_oracle(2)
    assert max_fluid_diff(case, fg, fo) <= TOL_F


# ---- neighbour indexing of the two-cell and staged kernels, checkpoint / resume, profiling env -----

@pytest.mark.parametrize("tma", [False, True])
@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
@pytest.mark.parametrize("dims, faces", [((32, 10, 7), (0, 0, 0)), ((2, 5, 3), (0, 0, 0)),
                                         ((22, 9, 4), (1, 1, 0)), ((48, 6, 5), (1, 0, 1))])
def test_streaming_permutation_bit_exact_two_cell(dims, faces, scheme, tma):
    """The permutation test on even nx (two cells per thread, x-wrap at both pair edges) and on nx
    a multiple of 16 (the staged odd step when tma): every label lands where the oracle puts it."""
    nx, ny, nz = dims
    r = np.random.default_rng(43)
    flags = (r.uniform(size=nx * ny * nz) < 0.2).astype(np.uint8)
    case = Case(nx, ny, nz, 1e30, wl.labels(nx * ny * nz), flags=flags, faces=faces)
    for steps in (1, 2, 5):
        fo, _ = case.run_oracle(steps)
        fg, _ = case.run_gpu(steps, "stream", scheme, tma=tma)
        fl = case.fluid
        assert np.array_equal(fg[:, fl], fo[:, fl]), steps


@pytest.mark.parametrize("scheme", ["AA", "AB", "AB2"])
def test_checkpoint_resume_across_parities(scheme):
    """lbm_get_populations + lbm_set_populations form a full checkpoint: stopping after an odd or an
    even number of steps (the AA buffer in either parity), restoring into a fresh context and
    continuing matches the uninterrupted run (to the rounding of f = (f - w) + w at the restore)."""
    case = mixed_case(24, 13, 9, (1, 0, 0), 1400, moving=0.3)
    total = 9
    full, _ = case.run_gpu(total, "stream", scheme)
    for k in (3, 4):
        ctx = case.gpu_context("stream", scheme)
        try:
            B.lbm_step(ctx, k)
            f = np.zeros((19, case.N), np.float32)
            B.lbm_get_populations(ctx, f)
        finally:
            B.lbm_destroy(ctx)
        resumed = Case(case.nx, case.ny, case.nz, case.tau, f, flags=case.flags, faces=case.faces,
                       inlet=case.inlet, g=case.g, wall=case.wall)
        fr, _ = resumed.run_gpu(total - k, "stream", scheme)
        assert max_fluid_diff(case, fr, full) <= 1e-6, k


def test_profile_environment_variable(monkeypatch):
    monkeypatch.setenv("LBM_PROFILE", "1")
    case = mixed_case(16, 8, 6, (0, 0, 0), 1500, inlet_layer=False)
    ctx = case.gpu_context("stream", "AA")
    try:
        B.lbm_step(ctx, 4)
        n_even, ms_even = B.lbm_profile_read(ctx, B.K_AA_EVEN)
        n_odd, _ = B.lbm_profile_read(ctx, B.K_AA_ODD)
        assert n_even == 2 and n_odd == 2 and ms_even > 0
    finally:
        B.lbm_destroy(ctx)
