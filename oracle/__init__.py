"""CPU oracle for the D3Q19 BGK step.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this package.  The
GPU library never calls it and shares no code with it.  The arithmetic lives in
``d3q19_oracle.cpp`` (plain loops, fp64); this module only builds it with g++ and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "d3q19_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

FLUID, SOLID, INLET, MOVING_WALL = 0, 1, 2, 3
PERIODIC, OPEN = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (g++, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        lib.oracle_tables.argtypes = [P, P, P]
        lib.oracle_equilibrium.argtypes = [d, P, P]
        lib.oracle_collide.argtypes = [P, d, P, P]
        lib.oracle_equilibrium_field.argtypes = [i64, P, P, P]
        lib.oracle_step_ab.argtypes = [i, i, i, d, P, P, P, P, P, P, i, P, i]
        lib.oracle_step_ab.restype = i
        lib.oracle_step_aa.argtypes = [i, i, i, d, P, P, P, P, P, P, i, i, P, i]
        lib.oracle_step_aa.restype = i
        lib.oracle_aa_natural.argtypes = [i, i, i, P, P, P, P, P, P]
        lib.oracle_aa_natural.restype = i
        lib.oracle_macroscopic.argtypes = [i, i, i, P, P, P, P, P, P, P]
        lib.oracle_macroscopic.restype = i
        lib.oracle_max_threads.restype = i
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        a = a.reshape(shape)
    return a


def tables():
    """(c[19,3] int, w[19] float64, opp[19] int) as the oracle defines them."""
    c = np.zeros((19, 3), np.int32)
    w = np.zeros(19, np.float64)
    opp = np.zeros(19, np.int32)
    _load().oracle_tables(_ptr(c), _ptr(w), _ptr(opp))
    return c, w, opp


def equilibrium(rho: float, u) -> np.ndarray:
    u = _f64(u, (3,))
    out = np.zeros(19, np.float64)
    _load().oracle_equilibrium(float(rho), _ptr(u), _ptr(out))
    return out


def collide(f, tau: float, g=(0.0, 0.0, 0.0)) -> np.ndarray:
    f = _f64(f, (19,))
    g = _f64(g, (3,))
    out = np.zeros(19, np.float64)
    _load().oracle_collide(_ptr(f), float(tau), _ptr(g), _ptr(out))
    return out


def equilibrium_field(rho, u) -> np.ndarray:
    """rho[N] (any shape), u[3, ...] -> f[19, N] natural SoA, fp64."""
    rho = _f64(rho).reshape(-1)
    N = rho.size
    u = _f64(u).reshape(3, N)
    f = np.zeros((19, N), np.float64)
    _load().oracle_equilibrium_field(N, _ptr(rho), _ptr(u), _ptr(f))
    return f


class Problem:
    """Grid, relaxation time, flags, faces, inlet state, body acceleration, wall velocity."""

    def __init__(self, nx, ny, nz, tau, flags=None, faces=(PERIODIC, PERIODIC, PERIODIC),
                 inlet=(1.0, 0.0, 0.0, 0.0), g=(0.0, 0.0, 0.0), threads=0,
                 wall=(0.0, 0.0, 0.0)):
        self.nx, self.ny, self.nz = int(nx), int(ny), int(nz)
        self.N = self.nx * self.ny * self.nz
        self.tau = float(tau)
        if flags is None:
            flags = np.zeros(self.N, np.uint8)
        self.flags = np.ascontiguousarray(flags, dtype=np.uint8).reshape(-1)
        assert self.flags.size == self.N
        self.faces = np.ascontiguousarray(faces, dtype=np.int32).reshape(3)
        self.inlet = _f64(inlet, (4,))
        self.g = _f64(g, (3,))
        self.wall = _f64(wall, (3,))
        self.threads = int(threads)

    def _args(self):
        return (self.nx, self.ny, self.nz, self.tau, _ptr(self.flags), _ptr(self.faces),
                _ptr(self.inlet), _ptr(self.g), _ptr(self.wall))

    def step_ab(self, f, nsteps: int, want_force: bool = False, inplace: bool = False):
        """Two-lattice steps on a copy of natural f[19, N]; returns (f_new, force or None).
        inplace=True updates f itself (a C-contiguous float64 array of 19 N values), which keeps
        the host memory of a large grid at two lattices instead of three."""
        if inplace:
            if not (isinstance(f, np.ndarray) and f.dtype == np.float64 and
                    f.flags["C_CONTIGUOUS"] and f.size == 19 * self.N):
                raise ValueError("inplace needs a C-contiguous float64 array of 19 N values")
            f = f.reshape(19, self.N)
        else:
            f = _f64(f).reshape(19, self.N).copy()
        force = np.zeros(3, np.float64) if want_force else None
        rc = _load().oracle_step_ab(*self._args(), _ptr(f), int(nsteps), _ptr(force),
                                    self.threads)
        if rc != 0:
            raise ValueError("oracle_step_ab: invalid arguments")
        return f, force

    def step_aa(self, A, parity: int, nsteps: int, want_force: bool = False):
        """In-place AA steps on a copy of buffer A[19, N]; returns (A_new, force or None)."""
        A = _f64(A).reshape(19, self.N).copy()
        force = np.zeros(3, np.float64) if want_force else None
        rc = _load().oracle_step_aa(*self._args(), _ptr(A), int(parity), int(nsteps),
                                    _ptr(force), self.threads)
        if rc != 0:
            raise ValueError("oracle_step_aa: invalid arguments")
        return A, force

    def aa_natural(self, A):
        A = _f64(A).reshape(19, self.N)
        f = np.zeros_like(A)
        rc = _load().oracle_aa_natural(self.nx, self.ny, self.nz, _ptr(self.flags),
                                       _ptr(self.faces), _ptr(self.inlet), _ptr(self.wall),
                                       _ptr(A), _ptr(f))
        if rc != 0:
            raise ValueError("oracle_aa_natural: invalid arguments")
        return f

    def macroscopic(self, f):
        f = _f64(f).reshape(19, self.N)
        rho = np.zeros(self.N, np.float64)
        u = np.zeros((3, self.N), np.float64)
        rc = _load().oracle_macroscopic(self.nx, self.ny, self.nz, _ptr(self.flags),
                                        _ptr(self.inlet), _ptr(self.wall), _ptr(self.g),
                                        _ptr(f), _ptr(rho), _ptr(u))
        if rc != 0:
            raise ValueError("oracle_macroscopic: invalid arguments")
        return rho, u


def max_threads() -> int:
    return int(_load().oracle_max_threads())
