"""CPU checks of the full-length oracle fixtures (tests/golden/full_*.npz) that the GPU tests in
test_gpu_full_length.py compare against: each fixture was written by the current oracle source
for the stated workload, samples only FLUID cells, and agrees with what physics fixes for it:

  * Taylor-Green 128^3 after 1000 steps (Reynolds number u0 / (nu k) ~ 30): the amplitude of the
    initial mode lies below its purely viscous decay exp(-3 nu k^2 t) (nu = (tau - 1/2)/3) --
    nonlinear transfer to other modes only drains it further -- and above 0.8 of it, and the u
    and v modes keep equal amplitudes (the lattice is symmetric under swapping x and y);
  * sphere 128^3 after 2000 steps: the drag points along the inflow and the transverse force
    vanishes by the mirror symmetry of the geometry about y = 64 and z = 64;
  * porous 512^3 after 500 steps from rest under g = 1e-6 along x: the mean velocity of the
    sampled cells points along g and stays below the free-fall value g t; the force on the solids
    points along g, stays below the total body force, and its transverse components are below 1%
    of it (the medium is statistically isotropic).
"""
import json
import math
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_full_length_goldens as G  # noqa: E402

from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl  # noqa: E402


def fixture(name):
    path = os.path.join(HERE, "golden", f"full_{name}.npz")
    if not os.path.exists(path):
        pytest.fail(f"missing fixture {path}: run tests/golden/make_full_length_goldens.py")
    z = np.load(path)
    return z, json.loads(str(z["meta"]))


@pytest.mark.parametrize("name", G.NAMES)
def test_fixture_matches_current_oracle_and_workload(name):
    z, meta = fixture(name)
    assert meta["oracle_hash"] == G.oracle_source_hash(), "oracle changed: regenerate the fixture"
    s = G.spec(name)
    assert meta["dims"] == list(s["dims"]) and meta["steps"] == s["steps"]
    assert meta["tau"] == s["tau"] and meta["g"] == list(s["g"])
    cells = z["cells"]
    assert cells.size >= G.SAMPLE
    assert np.all(np.diff(cells) > 0)
    assert np.all(s["flags"][cells] == wl.FLUID)
    S = cells.size
    assert z["f"].shape == (19, S) and z["rho"].shape == (S,) and z["u"].shape == (3, S)
    assert np.isfinite(z["f"]).all() and np.isfinite(z["force"]).all()
    # rho is the zeroth moment of the stored populations
    assert np.abs(z["f"].sum(axis=0) - z["rho"]).max() < 1e-12


def test_taylor_green_fixture_decays_at_the_viscous_rate():
    z, meta = fixture("taylor_green_128")
    n, tau, t = 128, meta["tau"], meta["steps"]
    nu = (tau - 0.5) / 3.0
    k = 2 * math.pi / n
    x, y, zz = wl.coords(n, n, n)
    c = z["cells"]
    mode_u = np.sin(k * x[c]) * np.cos(k * y[c]) * np.cos(k * zz[c])
    mode_v = -np.cos(k * x[c]) * np.sin(k * y[c]) * np.cos(k * zz[c])
    amp_u = float(np.dot(z["u"][0], mode_u) / np.dot(mode_u, mode_u))
    amp_v = float(np.dot(z["u"][1], mode_v) / np.dot(mode_v, mode_v))
    linear = 0.05 * math.exp(-3 * nu * k * k * t)
    assert 0.8 * linear < amp_u < linear, (amp_u, linear)
    assert abs(amp_v / amp_u - 1) < 5e-3, (amp_u, amp_v)
    # w starts at zero and is generated only by the nonlinear terms
    assert 0 < np.abs(z["u"][2]).max() < 0.5 * linear


def test_sphere_fixture_drag_is_along_the_flow_and_symmetric():
    z, _ = fixture("sphere_128")
    F = z["force"]
    assert F[0] > 0
    assert abs(F[1]) <= 1e-9 * F[0] and abs(F[2]) <= 1e-9 * F[0]


def test_porous_fixture_flow_follows_the_body_force():
    z, meta = fixture("porous_512")
    g, t = meta["g"][0], meta["steps"]
    ux = z["u"][0]
    assert 0 < ux.mean() < g * t
    F = z["force"]
    n = meta["dims"][0]
    total_body = g * n ** 3  # an upper bound: rho ~ 1 on at most every cell
    assert 0 < F[0] < total_body
    assert abs(F[1]) < 0.01 * F[0] and abs(F[2]) < 0.01 * F[0]
