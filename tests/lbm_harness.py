"""Helpers for the parity tests: run the same seeded problem through the CUDA library (via the
C ABI binding) and through the CPU oracle, and compare."""
from __future__ import annotations

import numpy as np

import oracle
from lattice_boltzmann_cfd_d3q19_gb300 import binding as B
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl

# max |f_gpu - f_oracle| over FLUID cells after N steps (fp32 GPU vs fp64 oracle, rho ~ 1)
TOL_F = 1e-5

LAYOUTS = {"stream": B.LAYOUT_STREAM, "bundle": B.LAYOUT_BUNDLE, "collision": B.LAYOUT_COLLISION}
# half-precision storage of the stream layout (its own tolerance, see fp16_tolerance)
FP16 = {"stream_fp16": B.LAYOUT_STREAM_FP16}


def fp16_tolerance(f0, steps, w=None):
    """Bound on |f_fp16 - f_fp32| after `steps` steps: every stored population is rounded to 11
    significant bits (relative error <= 2^-11) once when loaded and once per step; the collision
    mixes populations with weights of at most ~1, so the errors add at most linearly.  Twice that
    bound, on the largest shifted population |f - w| of the initial state."""
    import oracle
    if w is None:
        _, w, _ = oracle.tables()
    H = float(np.abs(np.asarray(f0, np.float64).reshape(19, -1) - w[:, None]).max())
    return 2.0 * (steps + 1) * H * 2.0 ** -11
SCHEMES = {"AA": B.STREAMING_AA, "AB": B.STREAMING_AB, "AB2": B.STREAMING_AB2}


class Case:
    """One problem: grid, tau, flags, faces, inlet, body force and initial natural state f0."""

    def __init__(self, nx, ny, nz, tau, f0, flags=None, faces=(0, 0, 0),
                 inlet=(1.0, 0.0, 0.0, 0.0), g=(0.0, 0.0, 0.0), wall=(0.0, 0.0, 0.0)):
        self.nx, self.ny, self.nz = nx, ny, nz
        self.N = nx * ny * nz
        self.tau = tau
        self.flags = np.zeros(self.N, np.uint8) if flags is None else np.asarray(flags, np.uint8)
        self.faces = tuple(faces)
        self.inlet = tuple(float(v) for v in inlet)
        self.g = tuple(float(v) for v in g)
        self.wall = tuple(float(v) for v in wall)
        # the input both sides start from, exactly representable in fp32
        if isinstance(f0, np.ndarray) and f0.dtype == np.float32:
            self.f0_32 = np.ascontiguousarray(f0.reshape(19, self.N))
        else:
            self.f0_32 = np.ascontiguousarray(np.asarray(f0, np.float64).reshape(19, self.N),
                                              dtype=np.float32)

    @property
    def fluid(self):
        return self.flags == wl.FLUID

    def oracle_problem(self, threads=0):
        return oracle.Problem(self.nx, self.ny, self.nz, self.tau, flags=self.flags,
                              faces=self.faces, inlet=self.inlet, g=self.g, threads=threads,
                              wall=self.wall)

    def run_oracle(self, steps, want_force=False):
        return self.oracle_problem().step_ab(self.f0_32.astype(np.float64), steps, want_force)

    def gpu_context(self, layout="stream", scheme="AA", device_input=True, pairs=True, tma=False,
                    overlap=True):
        import torch
        ctx = B.lbm_create(self.nx, self.ny, self.nz, self.tau, {**LAYOUTS, **FP16}[layout],
                           SCHEMES[scheme])
        try:
            B.lbm_set_cell_pairs(ctx, pairs)
            B.lbm_set_tma_gather(ctx, tma)
            B.lbm_set_boundary_overlap(ctx, overlap)
            B.lbm_set_flags(ctx, self.flags)
            B.lbm_set_faces(ctx, *self.faces)
            B.lbm_set_inlet(ctx, *self.inlet)
            B.lbm_set_body_force(ctx, *self.g)
            B.lbm_set_wall_velocity(ctx, *self.wall)
            if device_input:
                B.lbm_set_populations(ctx, torch.from_numpy(self.f0_32.copy()).cuda())
            else:
                B.lbm_set_populations(ctx, self.f0_32)
        except Exception:
            B.lbm_destroy(ctx)
            raise
        return ctx

    def run_gpu(self, steps, layout="stream", scheme="AA", want_force=False, chunks=None,
                device_input=True, pairs=True, tma=False, overlap=True, graphs=True):
        """Returns (f[19, N] float64, force or None).  `chunks` splits the steps into several
        lbm_step calls (the force belongs to the last call).  pairs=False forbids the two-cell
        kernels, tma=True allows the TMA-staged odd step, overlap=False runs each boundary kernel
        after its main kernel, graphs=False launches kernel by kernel."""
        ctx = self.gpu_context(layout, scheme, device_input, pairs, tma, overlap)
        try:
            B.lbm_set_graph_launch(ctx, graphs)
            for n in (chunks or [steps]):
                B.lbm_step(ctx, n)
            f = np.zeros((19, self.N), np.float32)
            B.lbm_get_populations(ctx, f)
            F = B.lbm_force_momentum_exchange(ctx) if want_force and steps > 0 else None
        finally:
            B.lbm_destroy(ctx)
        return f.astype(np.float64), F


def max_fluid_diff(case, fa, fb):
    fl = case.fluid
    if not fl.any():
        return 0.0
    return float(np.abs(fa[:, fl] - fb[:, fl]).max())


def random_state(N, seed, amp=1e-2, du=0.05):
    r = np.random.default_rng(seed)
    rho = 1 + r.uniform(-0.05, 0.05, N)
    u = r.uniform(-du, du, (3, N))
    f = oracle.equilibrium_field(rho, u)
    return f * (1 + amp * r.uniform(-1, 1, f.shape))


def window(case, center, half, f):
    """Sub-problem of side 2*half+1 around `center` (periodic wrap in the full domain), with the
    flags and state of the full problem, periodic on its own faces.  After at most `half` steps
    its central cell equals the full problem's (light cone of the nearest-neighbour stencil)."""
    nx, ny, nz = case.nx, case.ny, case.nz
    cxx, cyy, czz = center
    d = np.arange(-half, half + 1)
    xs, ys, zs = (cxx + d) % nx, (cyy + d) % ny, (czz + d) % nz
    idx = (xs[None, None, :] + nx * (ys[None, :, None] + ny * zs[:, None, None])).reshape(-1)
    m = 2 * half + 1
    sub = Case(m, m, m, case.tau, f.reshape(19, -1)[:, idx], flags=case.flags[idx],
               inlet=case.inlet, g=case.g, wall=case.wall)
    centre_index = half + m * (half + m * half)
    return sub, centre_index, idx
