"""Pins of the CPU oracle to facts fixed by the pages and by mathematics (no GPU involved).

Each test checks the oracle against something other than itself: exact rational moments, closed
forms (equilibrium moments, Taylor-Green decay, Poiseuille flow), conservation laws, symmetry, a
forward particle tracer, and the equivalence of two independently written streaming schemes.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl


def frac_weights():
    c, w, opp = oracle.tables()
    return c, [Fraction(x).limit_denominator(1000) for x in w], w, opp


# ---- velocity set and weights ---------------------------------------------------------------

def test_velocity_set_and_weights_match_page(golden):
    c, wf, w, opp = frac_weights()
    vel = {tuple(v) for v in c.tolist()}
    expect = {(0, 0, 0)}
    for a in range(3):
        for s in (1, -1):
            e = [0, 0, 0]
            e[a] = s
            expect.add(tuple(e))
    for a in range(3):
        for b in range(a + 1, 3):
            for sa in (1, -1):
                for sb in (1, -1):
                    e = [0, 0, 0]
                    e[a], e[b] = sa, sb
                    expect.add(tuple(e))
    assert len(vel) == 19 and vel == expect
    by_class = {int(r[1]): (int(r[2]), Fraction(int(r[3]), int(r[4])))
                for r in golden("d3q19_weights.txt")}
    for s2, (count, weight) in by_class.items():
        members = [q for q in range(19) if int((c[q] ** 2).sum()) == s2]
        assert len(members) == count
        for q in members:
            assert wf[q] == weight
            assert abs(w[q] - float(weight)) < 1e-16
    for q in range(19):
        assert (c[opp[q]] == -c[q]).all()


def test_isotropy_moments_exact():
    """sum w = 1, sum w c = 0, sum w c c = I/3, sum w ccc = 0, sum w cccc = (dd+dd+dd)/9."""
    c, wf, _, _ = frac_weights()
    d = lambda i, j: 1 if i == j else 0
    assert sum(wf) == 1
    for a in range(3):
        assert sum(wf[q] * c[q][a] for q in range(19)) == 0
        for b in range(3):
            assert sum(wf[q] * c[q][a] * c[q][b] for q in range(19)) == Fraction(d(a, b), 3)
            for g in range(3):
                assert sum(wf[q] * c[q][a] * c[q][b] * c[q][g] for q in range(19)) == 0
                for e in range(3):
                    m4 = sum(wf[q] * c[q][a] * c[q][b] * c[q][g] * c[q][e] for q in range(19))
                    expect = Fraction(d(a, b) * d(g, e) + d(a, g) * d(b, e) + d(a, e) * d(b, g),
                                      9)
                    assert m4 == expect


# ---- equilibrium and collision ----------------------------------------------------------------

def test_equilibrium_moments():
    c, _, _, _ = frac_weights()
    r = np.random.default_rng(7)
    for _ in range(20):
        rho = r.uniform(0.5, 1.5)
        u = r.uniform(-0.1, 0.1, 3)
        feq = oracle.equilibrium(rho, u)
        assert abs(feq.sum() - rho) < 1e-15
        assert np.abs(c.T @ feq - rho * u).max() < 1e-15
        Pi = np.einsum("q,qa,qb->ab", feq, c, c)
        assert np.abs(Pi - (rho / 3 * np.eye(3) + rho * np.outer(u, u))).max() < 1e-15


def test_equilibrium_is_fixed_point_of_collision():
    r = np.random.default_rng(8)
    for tau in (0.51, 0.6, 1.0, 1.7):
        rho, u = r.uniform(0.8, 1.2), r.uniform(-0.05, 0.05, 3)
        feq = oracle.equilibrium(rho, u)
        assert np.abs(oracle.collide(feq, tau) - feq).max() < 4 * np.finfo(float).eps


def test_collision_relaxes_nonequilibrium_by_one_minus_omega():
    """f* - f_eq = (1 - 1/tau) (f - f_eq) with g = 0 (PortLBM Eq. 1)."""
    r = np.random.default_rng(9)
    rho, u = 1.02, np.array([0.03, -0.01, 0.02])
    feq = oracle.equilibrium(rho, u)
    c, _, _, _ = frac_weights()
    # a perturbation with zero mass and momentum keeps rho and u, hence f_eq
    p = r.normal(size=19) * 1e-3
    M = np.vstack([np.ones(19), c.T.astype(float)])
    p -= M.T @ np.linalg.lstsq(M.T, p, rcond=None)[0]
    f = feq + p
    tau = 0.73
    post = oracle.collide(f, tau)
    assert np.abs((post - feq) - (1 - 1 / tau) * p).max() < 1e-15


def test_guo_source_moments():
    """With g != 0: mass is unchanged and momentum grows by exactly rho g per collision."""
    c, _, _, _ = frac_weights()
    r = np.random.default_rng(10)
    f = oracle.equilibrium(1.05, [0.01, 0.02, -0.03]) + r.normal(size=19) * 1e-4
    g = np.array([1e-3, -2e-3, 5e-4])
    post = oracle.collide(f, 0.8, g)
    rho = f.sum()
    assert abs(post.sum() - rho) < 1e-15
    assert np.abs(c.T @ post - (c.T @ f + rho * g)).max() < 1e-15


def test_guo_equals_shifted_velocity_relaxation_plus_constant():
    """The forcing identity the GPU collision uses: with a quadratic equilibrium, the literal Guo
    collision equals BGK relaxation toward f_eq(j/rho + tau g) plus
    -omega (tau - 1/2)^2 w rho (4.5 (c.g)^2 - 1.5 g.g) per population."""
    c, _, w, _ = frac_weights()
    r = np.random.default_rng(12)
    for tau in (0.55, 0.7, 1.3):
        om, a = 1 / tau, tau - 0.5
        g = r.uniform(-1e-3, 1e-3, 3)
        f = oracle.equilibrium(1.03, [0.02, -0.01, 0.03]) + r.normal(size=19) * 1e-4
        rho = f.sum()
        j = c.T.astype(float) @ f
        feq = oracle.equilibrium(rho, j / rho + tau * g)
        cg = c.astype(float) @ g
        alt = f - om * (f - feq) - om * a * a * w * rho * (4.5 * cg ** 2 - 1.5 * g @ g)
        assert np.abs(alt - oracle.collide(f, tau, g)).max() < 1e-15


# ---- whole-lattice invariants ----------------------------------------------------------------

def random_state(N, seed, amp=1e-2):
    r = np.random.default_rng(seed)
    rho = 1 + r.uniform(-0.05, 0.05, N)
    u = r.uniform(-0.05, 0.05, (3, N))
    f = oracle.equilibrium_field(rho, u)
    return f * (1 + amp * r.uniform(-1, 1, f.shape))


def test_uniform_flow_stays_uniform():
    P = oracle.Problem(6, 5, 4, 0.7)
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N, 1.01, (0.04, -0.02, 0.01)))
    f, _ = P.step_ab(f0, 7)
    assert np.abs(f - f0).max() < 4 * np.finfo(float).eps


@pytest.mark.parametrize("g", [(0, 0, 0), (1e-4, -3e-5, 2e-5)])
def test_mass_and_momentum_conservation_periodic(g):
    c, _, _, _ = frac_weights()
    P = oracle.Problem(7, 6, 5, 0.65, g=g)
    f = random_state(P.N, 11)
    mass0 = f.sum()
    mom0 = (c.T.astype(float) @ f).sum(axis=1)
    for t in range(1, 13):
        f, _ = P.step_ab(f, 1)
        assert abs(f.sum() / mass0 - 1) < 1e-13
        mom = (c.T.astype(float) @ f).sum(axis=1)
        assert np.abs(mom - (mom0 + t * mass0 * np.asarray(g))).max() < 1e-12 * mass0


def test_mass_conserved_with_walls():
    P = oracle.Problem(5, 8, 4, 0.9, flags=wl.channel_flags(5, 8, 4), g=(1e-4, 0, 0))
    fl = P.flags == wl.FLUID
    f = random_state(P.N, 12)
    m0 = f[:, fl].sum()
    f, _ = P.step_ab(f, 25)
    assert abs(f[:, fl].sum() / m0 - 1) < 1e-13


# ---- Taylor-Green decay (nu = (tau - 1/2)/3, GPU加速LBM §5.1) --------------------------------

def mode_amplitude(P, f, shape):
    rho, u = P.macroscopic(f)
    return float((u[0] * shape).sum() / (shape * shape).sum())


def test_taylor_green_2d_decay_rate():
    n, tau, u0 = 32, 0.6, 1e-3
    nu = (tau - 0.5) / 3
    k = 2 * math.pi / n
    P = oracle.Problem(n, n, 1, tau)
    rho, u = wl.taylor_green(n, n, 1, u0, two_d=True)
    x, y, _ = wl.coords(n, n, 1)
    shape = np.sin(k * x) * np.cos(k * y)
    f, _ = P.step_ab(oracle.equilibrium_field(rho, u), 100)
    a1 = mode_amplitude(P, f, shape)
    f, _ = P.step_ab(f, 500)
    a2 = mode_amplitude(P, f, shape)
    rate = -math.log(a2 / a1) / 500
    assert abs(rate / (2 * nu * k * k) - 1) < 0.01


def test_taylor_green_3d_decay_rate():
    n, tau, u0 = 32, 0.6, 1e-3
    nu = (tau - 0.5) / 3
    k = 2 * math.pi / n
    P = oracle.Problem(n, n, n, tau)
    rho, u = wl.taylor_green(n, n, n, u0)
    x, y, z = wl.coords(n, n, n)
    shape = np.sin(k * x) * np.cos(k * y) * np.cos(k * z)
    f, _ = P.step_ab(oracle.equilibrium_field(rho, u), 40)
    a1 = mode_amplitude(P, f, shape)
    f, _ = P.step_ab(f, 200)
    a2 = mode_amplitude(P, f, shape)
    rate = -math.log(a2 / a1) / 200
    assert abs(rate / (3 * nu * k * k) - 1) < 0.02


# ---- Poiseuille flow between halfway bounce-back walls ------------------------------------------

def poiseuille_transient(eta, t, g, nu, H, terms=200):
    u = g / (2 * nu) * eta * (H - eta)
    for m in range(1, 2 * terms, 2):
        u -= (4 * g * H * H / (nu * math.pi ** 3 * m ** 3)) * np.sin(m * math.pi * eta / H) \
            * math.exp(-m * m * math.pi ** 2 * nu * t / (H * H))
    return u


def channel_run(ny, tau, g, steps, nx=1, nz=1):
    P = oracle.Problem(nx, ny, nz, tau, flags=wl.channel_flags(nx, ny, nz), g=(g, 0, 0))
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N))
    f, F = P.step_ab(f0, steps, want_force=True)
    return P, f, F


def test_poiseuille_transient_profile():
    ny, tau, g, steps = 64, 0.8, 1e-6, 20000
    nu, H = (tau - 0.5) / 3, ny - 2
    P, f, _ = channel_run(ny, tau, g, steps)
    _, u = P.macroscopic(f)
    y = np.arange(1, ny - 1)
    ux = u[0][1:ny - 1]
    expect = poiseuille_transient(y - 0.5, steps, g, nu, H)
    umax = g * H * H / (8 * nu)
    assert abs(umax - 4.805e-3) < 1e-5
    assert np.abs(ux - expect).max() < 0.01 * umax


def test_poiseuille_steady_state_and_wall_force_balance():
    """At tau = 1/2 + sqrt(3)/4 halfway bounce-back puts the wall exactly mid-link for BGK, so the
    steady profile is the parabola; the wall force balances the total body force."""
    ny, g = 24, 1e-5
    tau = 0.5 + math.sqrt(3) / 4
    nu, H = (tau - 0.5) / 3, ny - 2
    P, f, F = channel_run(ny, tau, g, 60000)
    rho, u = P.macroscopic(f)
    y = np.arange(1, ny - 1)
    expect = g / (2 * nu) * (y - 0.5) * (H - (y - 0.5))
    assert np.abs(u[0][1:ny - 1] - expect).max() < 1e-6 * expect.max()
    total_body = g * rho[P.flags == wl.FLUID].sum()
    assert abs(F[0] / total_body - 1) < 1e-6
    assert abs(F[1]) < 1e-12 and abs(F[2]) < 1e-12


def test_channel_reduces_to_one_column():
    """An x/z-invariant channel evolves identically on 4x16x3 and on 1x16x1 (bit-exact)."""
    Pa, fa, Fa = channel_run(16, 0.8, 1e-5, 50, nx=4, nz=3)
    Pb, fb, Fb = channel_run(16, 0.8, 1e-5, 50)
    fa = fa.reshape(19, 3, 16, 4)
    for z in range(3):
        for x in range(4):
            assert np.array_equal(fa[:, z, :, x], fb.reshape(19, 16))
    assert np.abs(Fa - Fb * 12).max() < 1e-11 * abs(Fa[0])


# ---- open face, inlet, bounce-back geometry ------------------------------------------------------

def x_invariant_state(nx, ny, nz, seed):
    f1 = random_state(ny * nz, seed).reshape(19, nz, ny, 1)
    return np.broadcast_to(f1, (19, nz, ny, nx)).reshape(19, -1).copy()


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_open_face_is_zero_gradient(axis):
    """A field invariant along an OPEN axis evolves exactly as with that axis PERIODIC."""
    n = [6, 5, 4]
    n[axis] = 5
    f = random_state(n[0] * n[1] * n[2], 13 + axis)
    f = f.reshape(19, n[2], n[1], n[0])
    sl = [slice(None)] * 4
    sl[3 - axis] = slice(0, 1)
    f = np.broadcast_to(f[tuple(sl)], f.shape).reshape(19, -1).copy()
    faces_open = [0, 0, 0]
    faces_open[axis] = 1
    g = (2e-5, -1e-5, 3e-5)
    Po = oracle.Problem(*n, 0.7, faces=faces_open, g=g)
    Pp = oracle.Problem(*n, 0.7, g=g)
    fo, _ = Po.step_ab(f, 9)
    fp, _ = Pp.step_ab(f, 9)
    assert np.array_equal(fo, fp)


@pytest.mark.parametrize("faces", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 0), (1, 1, 1)])
def test_open_face_ghost_layer_streaming(faces):
    """Collision off: streaming with OPEN faces equals streaming on a lattice padded with one
    ghost layer per open side that repeats the adjacent layer (edge padding), then cropped."""
    nx, ny, nz, steps = 5, 4, 6, 3
    c, _, _ = oracle.tables()
    P = oracle.Problem(nx, ny, nz, 1e30, faces=faces)
    f0 = wl.labels(P.N)
    f, _ = P.step_ab(f0, steps)
    F = f0.reshape(19, nz, ny, nx).copy()
    pad = [(1, 1) if faces[2 - k] else (0, 0) for k in range(3)]   # array axes z, y, x
    for _ in range(steps):
        new = np.empty_like(F)
        for q in range(19):
            G = np.pad(F[q], pad, mode="edge")
            # shift by c_q (periodic roll on closed axes, plain shift inside the padding)
            G = np.roll(G, shift=(c[q][2], c[q][1], c[q][0]), axis=(0, 1, 2))
            new[q] = G[tuple(slice(p0, G.shape[k] - p1) for k, (p0, p1) in enumerate(pad))]
        F = new
    assert np.array_equal(f, F.reshape(19, -1))


def test_inlet_feeds_its_equilibrium():
    """Fluid at f_eq(rho_in, u_in) next to an INLET layer and an OPEN outlet stays exactly there."""
    nx, ny, nz = 6, 4, 3
    u_in = (0.05, 0.01, -0.02)
    x, _, _ = wl.coords(nx, ny, nz)
    flags = np.where(x == 0, wl.INLET, wl.FLUID).astype(np.uint8)
    P = oracle.Problem(nx, ny, nz, 0.56, flags=flags, faces=(1, 0, 0), inlet=(1.0, *u_in))
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N, 1.0, u_in))
    f, _ = P.step_ab(f0, 11)
    fl = flags == wl.FLUID
    assert np.abs(f[:, fl] - f0[:, fl]).max() < 4 * np.finfo(float).eps


def trace_particles(nx, ny, nz, flags, steps):
    """Forward particle kinematics on a periodic lattice with halfway bounce-back: a particle at
    FLUID x moving with c_q goes to x + c_q if that cell is FLUID, otherwise it stays at x with
    the reversed velocity.  Returns dest[(q, n)] -> (q', n') after `steps` moves."""
    c, _, opp = oracle.tables()
    def cell(x, y, z):
        return (x % nx) + nx * ((y % ny) + ny * (z % nz))
    X, Y, Z = wl.coords(nx, ny, nz)
    dest = {}
    for n in range(nx * ny * nz):
        if flags[n] != wl.FLUID:
            continue
        for q in range(19):
            cq, cn = q, n
            for _ in range(steps):
                x, y, z = X[cn], Y[cn], Z[cn]
                m = cell(x + c[cq][0], y + c[cq][1], z + c[cq][2])
                if flags[m] == wl.FLUID:
                    cn = m
                else:
                    cq = int(opp[cq])
            dest[(q, n)] = (cq, cn)
    return dest


@pytest.mark.parametrize("steps", [1, 2, 5])
def test_streaming_permutation_bit_exact(steps):
    """With collision switched off (tau -> infinity, g = 0) a step only moves populations: the
    oracle must carry every integer label to where forward particle tracing puts it."""
    nx, ny, nz = 5, 6, 4
    r = np.random.default_rng(21)
    flags = (r.uniform(size=nx * ny * nz) < 0.25).astype(np.uint8)
    P = oracle.Problem(nx, ny, nz, 1e30, flags=flags)
    f0 = wl.labels(P.N)
    f, _ = P.step_ab(f0, steps)
    dest = trace_particles(nx, ny, nz, flags, steps)
    for (q, n), (q2, n2) in dest.items():
        assert f[q2, n2] == f0[q, n]
    # AA in-place reaches the same permutation
    A, _ = P.step_aa(f0, 0, steps)
    fa = P.aa_natural(A) if steps % 2 else A
    fl = flags == wl.FLUID
    assert np.array_equal(fa[:, fl], f[:, fl])


def test_streaming_periodic_shift_closed_form():
    """No solids, collision off: f_q(x, t) = f_q(x - t c_q, 0)."""
    nx, ny, nz, steps = 7, 5, 6, 4
    c, _, _ = oracle.tables()
    P = oracle.Problem(nx, ny, nz, 1e30)
    f0 = wl.labels(P.N)
    f, _ = P.step_ab(f0, steps)
    F0 = f0.reshape(19, nz, ny, nx)
    F = f.reshape(19, nz, ny, nx)
    for q in range(19):
        shifted = np.roll(F0[q], shift=(steps * c[q][2], steps * c[q][1], steps * c[q][0]),
                          axis=(0, 1, 2))
        assert np.array_equal(F[q], shifted)


# ---- AA in place == two lattices (GPU lattice Boltzmann: streaming layout, "In place") ---------

AA_CASES = [
    # nx, ny, nz, faces, solid fraction, inlet layer, g
    (5, 4, 3, (0, 0, 0), 0.0, False, (0, 0, 0)),
    (6, 5, 4, (0, 0, 0), 0.3, False, (1e-4, 0, -2e-5)),
    (6, 5, 4, (1, 0, 0), 0.2, True, (0, 0, 0)),
    (5, 6, 4, (1, 1, 0), 0.15, True, (3e-5, 2e-5, 0)),
    (4, 5, 6, (1, 1, 1), 0.2, False, (0, 0, 1e-5)),
    (3, 3, 3, (0, 1, 1), 0.25, True, (0, 0, 0)),
    (6, 5, 4, (1, 0, 0), 0.3, True, (2e-5, 0, 0)),   # with moving walls (see below)
]
MOVING_CASES = {6}


@pytest.mark.parametrize("case", range(len(AA_CASES)))
@pytest.mark.parametrize("steps", [1, 2, 3, 6])
def test_aa_in_place_equals_two_lattice(case, steps):
    nx, ny, nz, faces, solid, inlet_layer, g = AA_CASES[case]
    r = np.random.default_rng(100 + case)
    N = nx * ny * nz
    flags = (r.uniform(size=N) < solid).astype(np.uint8)
    if inlet_layer:
        x, _, _ = wl.coords(nx, ny, nz)
        flags[x == 0] = wl.INLET
    if case in MOVING_CASES:
        flags[(flags == wl.SOLID) & (r.uniform(size=N) < 0.5)] = wl.MOVING_WALL
    P = oracle.Problem(nx, ny, nz, 0.62, flags=flags, faces=faces,
                       inlet=(1.01, 0.03, -0.01, 0.02), g=g, wall=(0.03, -0.02, 0.01))
    f0 = random_state(N, 200 + case)
    fb, Fb = P.step_ab(f0, steps, want_force=True)
    A, Fa = P.step_aa(f0, 0, steps, want_force=True)
    fa = P.aa_natural(A) if steps % 2 else A
    fl = flags == wl.FLUID
    assert np.array_equal(fa[:, fl], fb[:, fl])
    assert np.array_equal(Fa, Fb)


# ---- momentum exchange --------------------------------------------------------------------------

def test_sphere_force_mirror_symmetry():
    nx, ny, nz = 16, 12, 12
    flags = wl.sphere_flags(nx, ny, nz, (6, 6, 6), 3, inlet_x0=False)
    P = oracle.Problem(nx, ny, nz, 0.7, flags=flags, g=(2e-5, 0, 0))
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N, 1.0, (0.02, 0, 0)))
    _, F = P.step_ab(f0, 30, want_force=True)
    assert F[0] > 0
    assert abs(F[1]) < 1e-12 * F[0] and abs(F[2]) < 1e-12 * F[0]


def test_force_counts_only_solid_links():
    """No solids -> zero force; one solid cell in a resting fluid -> the force is the sum of
    2 c_q w_q over its 18 links (rest state f* = w), which vanishes by symmetry."""
    P = oracle.Problem(4, 4, 4, 0.8)
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N))
    _, F = P.step_ab(f0, 1, want_force=True)
    assert np.array_equal(F, np.zeros(3))
    flags = np.zeros(P.N, np.uint8)
    flags[21] = wl.SOLID
    P2 = oracle.Problem(4, 4, 4, 0.8, flags=flags)
    _, F2 = P2.step_ab(f0, 1, want_force=True)
    assert np.abs(F2).max() < 1e-16
    # moving fluid pushes the cell downstream
    f1 = oracle.equilibrium_field(*wl.uniform_fields(P.N, 1.0, (0.05, 0, 0)))
    _, F3 = P2.step_ab(f1, 1, want_force=True)
    assert F3[0] > 0


def test_porous_generator_reaches_target():
    flags = wl.porous_flags(24, 20, 16, 0.30, 3, seed=5)
    frac = (flags == wl.SOLID).mean()
    assert 0.30 <= frac < 0.30 + 27 / flags.size + 1e-12
    again = wl.porous_flags(24, 20, 16, 0.30, 3, seed=5)
    assert np.array_equal(flags, again)


# ---- moving walls (GPU加速LBM §4.2 mirror method, reference density 1) ----------------------------

def couette(ny, tau, U, steps, nx=1, nz=1):
    flags = np.zeros(nx * ny * nz, np.uint8)
    _, y, _ = wl.coords(nx, ny, nz)
    flags[y == 0] = wl.SOLID
    flags[y == ny - 1] = wl.MOVING_WALL
    P = oracle.Problem(nx, ny, nz, tau, flags=flags, wall=(U, 0.0, 0.0))
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N))
    f, F = P.step_ab(f0, steps, want_force=True)
    return P, f, F


def test_couette_steady_profile_is_linear_and_wall_forces_balance():
    """Plane Couette flow between a resting wall (y = 0) and a wall moving at U (y = ny - 1):
    halfway bounce-back reproduces the linear profile u = U (y - 1/2) / H exactly, and at steady
    state the fluid's momentum no longer changes, so the forces on the two walls cancel."""
    ny, tau, U = 18, 0.9, 0.02
    H = ny - 2
    P, f, F = couette(ny, tau, U, 40000)
    rho, u = P.macroscopic(f)
    y = np.arange(1, ny - 1)
    assert np.abs(u[0][1:ny - 1] - U * (y - 0.5) / H).max() < 1e-9 * U
    assert np.abs(u[1:]).max() < 1e-12
    nu = (tau - 0.5) / 3
    assert abs(F[0]) < 1e-9 * nu * U / H   # resting wall gets +rho nu U/H, moving wall the opposite
    # shear stress from the non-equilibrium populations equals rho nu U / H in every fluid cell
    c, w, _ = oracle.tables()
    feq = oracle.equilibrium_field(rho, u)
    sxy = -(1 - 0.5 / tau) * ((c[:, 0] * c[:, 1])[:, None] * (f - feq)).sum(axis=0)
    assert np.abs(sxy[1:ny - 1] - nu * U / H).max() < 1e-6 * nu * U / H


def test_moving_wall_at_rest_equals_solid():
    nx, ny, nz = 6, 7, 5
    r = np.random.default_rng(31)
    flags = (r.uniform(size=nx * ny * nz) < 0.2).astype(np.uint8)
    moving = flags.copy()
    moving[moving == wl.SOLID] = wl.MOVING_WALL
    f0 = random_state(nx * ny * nz, 32)
    fs, Fs = oracle.Problem(nx, ny, nz, 0.7, flags=flags).step_ab(f0, 5, want_force=True)
    fm, Fm = oracle.Problem(nx, ny, nz, 0.7, flags=moving).step_ab(f0, 5, want_force=True)
    assert np.array_equal(fs, fm) and np.array_equal(Fs, Fm)


def test_lid_driven_cavity_conserves_mass():
    n = 10
    x, y, z = wl.coords(n, n, n)
    flags = np.zeros(n ** 3, np.uint8)
    flags[(x == 0) | (x == n - 1) | (y == 0) | (z == 0) | (z == n - 1)] = wl.SOLID
    flags[y == n - 1] = wl.MOVING_WALL
    P = oracle.Problem(n, n, n, 0.6, flags=flags, wall=(0.05, 0.0, 0.0))
    f0 = oracle.equilibrium_field(*wl.uniform_fields(P.N))
    fl = flags == wl.FLUID
    f, _ = P.step_ab(f0, 200)
    assert abs(f[:, fl].sum() / f0[:, fl].sum() - 1) < 1e-13
    _, u = P.macroscopic(f)
    assert u[0][fl].max() > 0.005          # the lid drags the fluid along
    # over one step the fluid's momentum changes by minus the momentum handed to the walls
    # (resting and moving) -- checks the moving-wall correction of the momentum exchange
    c, _, _ = oracle.tables()
    f2, F = P.step_ab(f, 1, want_force=True)
    dP = (c.T.astype(float) @ f2[:, fl]).sum(axis=1) - (c.T.astype(float) @ f[:, fl]).sum(axis=1)
    assert np.abs(dP + F).max() < 1e-13
