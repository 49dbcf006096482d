"""ctypes binding of liblbm.so: the C ABI of include/lbm.h under the same names.

Argument marshalling only -- every step of the computation runs in the library's CUDA kernels.
Arrays may be torch tensors (CUDA or CPU) or numpy arrays; they are passed as raw pointers and
must be C-contiguous with the dtype the C function expects.  A non-zero status raises LbmError
with the library's message.  The library must have been built (``build.build()``): there is no
fallback implementation, and loading fails loudly if liblbm.so is missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LAYOUT_STREAM, LAYOUT_BUNDLE, LAYOUT_COLLISION, LAYOUT_STREAM_FP16 = 0, 1, 2, 3
STREAMING_AUTO, STREAMING_AA, STREAMING_AB, STREAMING_AB2 = 0, 1, 2, 3
OK, EINVAL, ENOMEM, ECUDA, ESTATE, ENOTFINITE, ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
FLUID, SOLID, INLET, MOVING_WALL = 0, 1, 2, 3
PERIODIC, OPEN = 0, 1
# profiling kinds of lbm_profile_read
K_AA_EVEN, K_AA_ODD, K_AB_PULL, K_AB_COLLIDE, K_STREAM, K_PREGATHER, K_FORCE, K_BOUNDARY = range(8)

# every function declared in include/lbm.h, with (restype, argtypes)
_P, _I, _F, _D, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_int64
SIGNATURES = {
    "lbm_create": (_P, [_I, _I, _I, _F, _I, _I]),
    "lbm_last_error": (ctypes.c_char_p, []),
    "lbm_set_stream": (_I, [_P, _P]),
    "lbm_set_flags": (_I, [_P, _P]),
    "lbm_set_faces": (_I, [_P, _I, _I, _I]),
    "lbm_set_inlet": (_I, [_P, _F, _F, _F, _F]),
    "lbm_set_body_force": (_I, [_P, _F, _F, _F]),
    "lbm_set_wall_velocity": (_I, [_P, _F, _F, _F]),
    "lbm_set_populations": (_I, [_P, _P]),
    "lbm_set_equilibrium": (_I, [_P, _P, _P]),
    "lbm_get_populations": (_I, [_P, _P]),
    "lbm_step": (_I, [_P, _I]),
    "lbm_set_graph_launch": (_I, [_P, _I]),
    "lbm_set_cell_pairs": (_I, [_P, _I]),
    "lbm_set_tma_gather": (_I, [_P, _I]),
    "lbm_set_boundary_overlap": (_I, [_P, _I]),
    "lbm_macroscopic": (_I, [_P, _P, _P]),
    "lbm_force_momentum_exchange": (_I, [_P, _P]),
    "lbm_check_finite": (_I, [_P]),
    "lbm_step_count": (_I64, [_P]),
    "lbm_kernel_launches": (_I64, [_P]),
    "lbm_profile_enable": (_I, [_P, _I]),
    "lbm_profile_read": (_I, [_P, _I, _P, _P]),
    "lbm_destroy": (None, [_P]),
    "lbm_force_momentum_exchange_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _F,
                                                 _P, _P]),
    "lbm_set_ghost_planes": (_I, [_P, _I]),
    "lbm_halo_elements": (_I64, [_P]),
    "lbm_halo_element_bytes": (_I, [_P]),
    "lbm_halo_pack": (_I, [_P, _P, _P]),
    "lbm_halo_unpack": (_I, [_P, _P, _P]),
    "lbm_slab_step_begin": (_I, [_P, _P, _P]),
    "lbm_slab_step_end": (_I, [_P, _P, _P]),
}


class LbmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


_lib = None
# cells of every live context, so that array arguments can be checked against 19 N / 3 N / N
_cells = {}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load liblbm.so (building it first when missing).  Raises if it cannot be loaded."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(f"{_build.LIB} is missing: build it with "
                                   "python -m lattice_boltzmann_cfd_d3q19_gb300.build")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _err() -> str:
    msg = load().lbm_last_error()
    return msg.decode("utf-8", "replace") if msg else ""


def _check(rc: int) -> int:
    if rc != OK:
        raise LbmError(rc, _err())
    return rc


def _ptr(a, dtype, count=None) -> int:
    """Raw pointer of a torch tensor or numpy array with the given numpy dtype."""
    if a is None:
        raise ValueError("array argument is None")
    if hasattr(a, "data_ptr") and hasattr(a, "is_contiguous"):  # torch.Tensor
        import torch
        tdt = {np.float32: torch.float32, np.uint8: torch.uint8, np.float64: torch.float64}[dtype]
        if a.dtype != tdt:
            raise TypeError(f"expected {tdt}, got {a.dtype}")
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        if count is not None and a.numel() != count:
            raise ValueError(f"expected {count} elements, got {a.numel()}")
        return a.data_ptr()
    arr = a
    if not isinstance(arr, np.ndarray):
        raise TypeError("expected a torch tensor or a numpy array")
    if arr.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {arr.dtype}")
    if not arr.flags["C_CONTIGUOUS"]:
        raise ValueError("array must be C-contiguous")
    if count is not None and arr.size != count:
        raise ValueError(f"expected {count} elements, got {arr.size}")
    return arr.ctypes.data


# ---- the C ABI, same names -----------------------------------------------------------------------

def lbm_create(nx: int, ny: int, nz: int, tau: float, layout: int = LAYOUT_STREAM,
               streaming: int = STREAMING_AUTO) -> int:
    h = load().lbm_create(int(nx), int(ny), int(nz), float(tau), int(layout), int(streaming))
    if not h:
        raise LbmError(EINVAL, _err())
    _cells[h] = int(nx) * int(ny) * int(nz)
    return h


def _n(ctx: int, per_cell: int = 1):
    """Element count an array argument of this context must have (None for an unknown handle,
    which the library rejects itself)."""
    N = _cells.get(ctx)
    return None if N is None else per_cell * N


def lbm_last_error() -> str:
    return _err()


def lbm_set_stream(ctx: int, cuda_stream: int) -> None:
    _check(load().lbm_set_stream(ctx, cuda_stream))


def lbm_set_flags(ctx: int, flags) -> None:
    p = _ptr(flags, np.uint8, _n(ctx))
    _check(load().lbm_set_flags(ctx, p))


def lbm_set_faces(ctx: int, fx: int, fy: int, fz: int) -> None:
    _check(load().lbm_set_faces(ctx, int(fx), int(fy), int(fz)))


def lbm_set_inlet(ctx: int, rho: float, ux: float, uy: float, uz: float) -> None:
    _check(load().lbm_set_inlet(ctx, float(rho), float(ux), float(uy), float(uz)))


def lbm_set_body_force(ctx: int, gx: float, gy: float, gz: float) -> None:
    _check(load().lbm_set_body_force(ctx, float(gx), float(gy), float(gz)))


def lbm_set_wall_velocity(ctx: int, ux: float, uy: float, uz: float) -> None:
    _check(load().lbm_set_wall_velocity(ctx, float(ux), float(uy), float(uz)))


def lbm_set_populations(ctx: int, f) -> None:
    p = _ptr(f, np.float32, _n(ctx, 19))
    _check(load().lbm_set_populations(ctx, p))


def lbm_set_equilibrium(ctx: int, rho, u) -> None:
    pr, pu = _ptr(rho, np.float32, _n(ctx)), _ptr(u, np.float32, _n(ctx, 3))
    _check(load().lbm_set_equilibrium(ctx, pr, pu))


def lbm_get_populations(ctx: int, f) -> None:
    p = _ptr(f, np.float32, _n(ctx, 19))
    _check(load().lbm_get_populations(ctx, p))


def lbm_step(ctx: int, n: int) -> None:
    _check(load().lbm_step(ctx, int(n)))


def lbm_set_graph_launch(ctx: int, enable: bool) -> None:
    _check(load().lbm_set_graph_launch(ctx, 1 if enable else 0))


def lbm_set_cell_pairs(ctx: int, enable: bool) -> bool:
    """Allow or forbid the two-cell step kernels; True when they will run."""
    rc = load().lbm_set_cell_pairs(ctx, 1 if enable else 0)
    if rc < 0:
        raise LbmError(rc, _err())
    return rc == 1


def lbm_set_tma_gather(ctx: int, enable: bool) -> bool:
    """Allow or forbid the TMA-staged AA odd step; True when it will run."""
    rc = load().lbm_set_tma_gather(ctx, 1 if enable else 0)
    if rc < 0:
        raise LbmError(rc, _err())
    return rc == 1


def lbm_set_boundary_overlap(ctx: int, enable: bool) -> None:
    """Run each step's boundary kernel beside its main kernel (True) or after it (False)."""
    _check(load().lbm_set_boundary_overlap(ctx, 1 if enable else 0))


def lbm_macroscopic(ctx: int, rho, u) -> None:
    pr, pu = _ptr(rho, np.float32, _n(ctx)), _ptr(u, np.float32, _n(ctx, 3))
    _check(load().lbm_macroscopic(ctx, pr, pu))


def lbm_force_momentum_exchange(ctx: int) -> np.ndarray:
    F = np.zeros(3, np.float64)
    _check(load().lbm_force_momentum_exchange(ctx, F.ctypes.data))
    return F


def lbm_check_finite(ctx: int) -> bool:
    rc = load().lbm_check_finite(ctx)
    if rc == ENOTFINITE:
        return False
    _check(rc)
    return True


def lbm_step_count(ctx: int) -> int:
    return int(load().lbm_step_count(ctx))


def lbm_kernel_launches(ctx: int) -> int:
    return int(load().lbm_kernel_launches(ctx))


def lbm_profile_enable(ctx: int, enable: bool) -> None:
    _check(load().lbm_profile_enable(ctx, 1 if enable else 0))


def lbm_profile_read(ctx: int, kind: int):
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(load().lbm_profile_read(ctx, int(kind), ctypes.addressof(n), ctypes.addressof(ms)))
    return int(n.value), float(ms.value)


def lbm_destroy(ctx: int) -> None:
    if ctx:
        _cells.pop(ctx, None)
        load().lbm_destroy(ctx)


def lbm_set_ghost_planes(ctx: int, enable: bool) -> None:
    _check(load().lbm_set_ghost_planes(ctx, 1 if enable else 0))


def lbm_halo_elements(ctx: int) -> int:
    return int(load().lbm_halo_elements(ctx))


def lbm_halo_element_bytes(ctx: int) -> int:
    rc = load().lbm_halo_element_bytes(ctx)
    if rc < 0:
        raise LbmError(rc, _err())
    return int(rc)


def _halo_ptr(ctx: int, t) -> int:
    """A halo buffer: a contiguous CUDA tensor of lbm_halo_elements values of the stored width."""
    import torch
    width = lbm_halo_element_bytes(ctx)
    want = torch.float16 if width == 2 else torch.float32
    if not (hasattr(t, "data_ptr") and t.is_cuda and t.is_contiguous()):
        raise ValueError("halo buffers are contiguous CUDA tensors")
    if t.dtype != want or t.numel() != lbm_halo_elements(ctx):
        raise ValueError(f"halo buffer must hold {lbm_halo_elements(ctx)} {want} values")
    return t.data_ptr()


def lbm_halo_pack(ctx: int, lo, hi) -> None:
    pl, ph = _halo_ptr(ctx, lo), _halo_ptr(ctx, hi)
    _check(load().lbm_halo_pack(ctx, pl, ph))


def lbm_halo_unpack(ctx: int, from_below, from_above) -> None:
    pb, pa = _halo_ptr(ctx, from_below), _halo_ptr(ctx, from_above)
    _check(load().lbm_halo_unpack(ctx, pb, pa))


def lbm_slab_step_begin(ctx: int, lo, hi) -> None:
    pl, ph = _halo_ptr(ctx, lo), _halo_ptr(ctx, hi)
    _check(load().lbm_slab_step_begin(ctx, pl, ph))


def lbm_slab_step_end(ctx: int, from_below, from_above) -> None:
    pb, pa = _halo_ptr(ctx, from_below), _halo_ptr(ctx, from_above)
    _check(load().lbm_slab_step_end(ctx, pb, pa))


def lbm_force_momentum_exchange_noalloc(f, flags, nx: int, ny: int, nz: int, faces=(0, 0, 0),
                                        tau: float = 0.6, g=(0.0, 0.0, 0.0),
                                        cuda_stream: int = 0) -> np.ndarray:
    """Force of one collision of the device state f with no allocation (see include/lbm.h).
    f must hold 19 nx ny nz floats and flags nx ny nz bytes: the C side cannot check array sizes,
    so they are checked here before the call."""
    N = int(nx) * int(ny) * int(nz)
    pf = _ptr(f, np.float32, count=19 * N)
    pflags = _ptr(flags, np.uint8, count=N)
    F = np.zeros(3, np.float64)
    _check(load().lbm_force_momentum_exchange_noalloc(
        pf, pflags, int(nx), int(ny), int(nz), int(faces[0]), int(faces[1]), int(faces[2]),
        float(tau), float(g[0]), float(g[1]), float(g[2]), F.ctypes.data, cuda_stream or None))
    return F
