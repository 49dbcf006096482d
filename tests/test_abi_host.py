"""Host-side checks of the C ABI (no GPU needed): the library loads and exports every function
include/lbm.h declares, and argument validation that happens before any CUDA call."""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

from lattice_boltzmann_cfd_d3q19_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "lbm.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lbm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = header_functions()
    for required in ("lbm_create", "lbm_set_populations", "lbm_step", "lbm_macroscopic",
                     "lbm_force_momentum_exchange", "lbm_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = B.load()
    for name in header_functions():
        assert hasattr(lib, name), name
    assert set(header_functions()) == set(B.SIGNATURES)


def test_library_symbols_with_nm():
    B.load()
    out = subprocess.run(["nm", "-D", "--defined-only", B.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (lbm_[a-z_0-9]+)$", out, flags=re.M))
    assert set(header_functions()) <= exported


@pytest.mark.parametrize("args, fragment", [
    ((0, 4, 4, 0.6, 0, 0), "extent"),
    ((4, -1, 4, 0.6, 0, 0), "extent"),
    ((4, 4, 4, 0.5, 0, 0), "tau"),
    ((4, 4, 4, float("nan"), 0, 0), "tau"),
    ((4, 4, 4, float("inf"), 0, 0), "tau"),
    ((4, 4, 4, 0.6, 4, 0), "layout"),
    ((4, 4, 4, 0.6, 0, 4), "streaming"),
    ((4, 70000, 4, 0.6, 0, 0), "65535"),
    ((2048, 2048, 1024, 0.6, 0, 0), "2^31"),
])
def test_create_rejects_invalid_arguments(args, fragment):
    with pytest.raises(B.LbmError) as ei:
        B.lbm_create(*args)
    assert fragment in str(ei.value)


def test_null_context_calls_fail_cleanly():
    lib = B.load()
    assert lib.lbm_step(None, 1) == B.EINVAL
    assert "NULL" in B.lbm_last_error()
    assert lib.lbm_set_faces(None, 0, 0, 0) == B.EINVAL
    assert lib.lbm_set_inlet(None, 1.0, 0.0, 0.0, 0.0) == B.EINVAL
    assert lib.lbm_set_body_force(None, 0.0, 0.0, 0.0) == B.EINVAL
    assert lib.lbm_check_finite(None) == B.EINVAL
    assert lib.lbm_set_cell_pairs(None, 1) == B.EINVAL
    assert lib.lbm_set_tma_gather(None, 1) == B.EINVAL
    assert lib.lbm_set_boundary_overlap(None, 1) == B.EINVAL
    assert lib.lbm_set_graph_launch(None, 1) == B.EINVAL
    assert lib.lbm_step_count(None) == -1
    assert lib.lbm_kernel_launches(None) == -1
    # the slab-decomposition calls
    assert lib.lbm_set_ghost_planes(None, 1) == B.EINVAL
    assert lib.lbm_halo_elements(None) == -1
    assert lib.lbm_halo_element_bytes(None) == B.EINVAL
    assert lib.lbm_halo_pack(None, None, None) == B.EINVAL
    assert lib.lbm_halo_unpack(None, None, None) == B.EINVAL
    assert lib.lbm_slab_step_begin(None, None, None) == B.EINVAL
    assert lib.lbm_slab_step_end(None, None, None) == B.EINVAL
    lib.lbm_destroy(None)  # NULL-safe


def test_allocation_failure_hook_reports_enomem():
    code = ("import lattice_boltzmann_cfd_d3q19_gb300.binding as B\n"
            "try:\n    B.lbm_create(4, 4, 4, 0.6)\nexcept B.LbmError as e:\n    print(e)\n")
    env = dict(os.environ, LBM_FAIL_ALLOC="1", PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         cwd=ROOT).stdout
    assert "allocation refused" in out


def test_binding_rejects_wrong_dtype_and_layout():
    a = np.zeros(10, np.float64)
    with pytest.raises(TypeError):
        B._ptr(a, np.float32)
    b = np.zeros((4, 4), np.float32)[:, ::2]
    with pytest.raises(ValueError):
        B._ptr(b, np.float32)


def test_shifted_storage_round_trips_integer_labels():
    """The library stores f - w in fp32; for the integer labels of the streaming-permutation test
    fl(fl(L - w) + w) == L must hold for every label and weight (checked in numpy fp32)."""
    L = np.arange(1, 19 * 32 ** 3 + 20, dtype=np.float32)
    for w in (np.float32(1 / 3), np.float32(1 / 18), np.float32(1 / 36)):
        h = (L - w).astype(np.float32)
        assert np.array_equal((h + w).astype(np.float32), L)


def test_noalloc_binding_checks_array_sizes_before_the_call():
    """The C side cannot see array sizes: the binding rejects a population array shorter than
    19 nx ny nz floats or a flag array shorter than nx ny nz bytes before calling into the
    library (a short array would otherwise be read past its end on the device)."""
    with pytest.raises(ValueError):
        B.lbm_force_momentum_exchange_noalloc(np.zeros(19 * 8 - 1, np.float32),
                                              np.zeros(8, np.uint8), 2, 2, 2)
    with pytest.raises(ValueError):
        B.lbm_force_momentum_exchange_noalloc(np.zeros(19 * 8, np.float32),
                                              np.zeros(7, np.uint8), 2, 2, 2)


def test_context_binding_checks_array_sizes():
    """Arrays passed with a context are checked against its cell count (19 N populations, N
    flags or densities, 3 N velocities) before the call."""
    ctx = 12345  # a handle the binding knows; no call reaches the library
    B._cells[ctx] = 8
    try:
        for fn, args in ((B.lbm_set_populations, (np.zeros(19 * 8 + 1, np.float32),)),
                         (B.lbm_get_populations, (np.zeros(19 * 7, np.float32),)),
                         (B.lbm_set_flags, (np.zeros(9, np.uint8),)),
                         (B.lbm_macroscopic, (np.zeros(8, np.float32), np.zeros(23, np.float32))),
                         (B.lbm_set_equilibrium, (np.zeros(7, np.float32),
                                                  np.zeros(24, np.float32)))):
            with pytest.raises(ValueError):
                fn(ctx, *args)
    finally:
        B._cells.pop(ctx, None)
