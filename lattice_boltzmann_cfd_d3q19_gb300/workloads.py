"""Seeded synthetic inputs for the D3Q19 workloads: macroscopic fields and cell-flag arrays.

This module holds no lattice Boltzmann arithmetic (no equilibrium, collision or streaming): it
only builds density / velocity fields and geometry, with numpy's PCG64 generator, so that the GPU
library and the CPU oracle are fed identical inputs.  Cell index n = x + nx*(y + ny*z); fields are
returned flat (rho[N], u[3, N]) in float64; flags are uint8 (0 fluid, 1 solid, 2 inlet,
3 moving wall).

Workloads (sizes as named by their callers):
  * Taylor-Green vortex (the validation case PortLBM lists beside Hagen-Poiseuille and Karman
    streets): u = u0 sin(kx) cos(ky) cos(kz), v = -u0 cos(kx) sin(ky) cos(kz), w = 0, k = 2 pi / n
    per axis, at integer cell coordinates; rho = 1 + U(-a, a).
  * channel: bounce-back walls on the layers y = 0 and y = ny - 1.
  * sphere: SOLID where (x-cx)^2 + (y-cy)^2 + (z-cz)^2 <= r^2, optional INLET layer at x = 0.
  * porous medium: 3x3x3 solid blobs at uniformly drawn corners (periodic wrap), drawn in order
    until the solid fraction first reaches the target.
  * lid-driven cavity: resting walls on five faces, a moving lid (MOVING_WALL) on the sixth.
"""
from __future__ import annotations

import math

import numpy as np

FLUID, SOLID, INLET, MOVING_WALL = 0, 1, 2, 3

# seed of each named workload: 1000 + its position in the list of workloads
SEED_TG32 = 1001
SEED_CHANNEL64 = 1002
SEED_TG128 = 1003
SEED_SPHERE128 = 1004
SEED_POROUS512 = 1005


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def coords(nx: int, ny: int, nz: int):
    """Integer coordinates (x, y, z) of every cell, flat in cell-index order."""
    n = np.arange(nx * ny * nz, dtype=np.int64)
    return n % nx, (n // nx) % ny, n // (nx * ny)


def uniform_fields(N: int, rho: float = 1.0, u=(0.0, 0.0, 0.0)):
    r = np.full(N, float(rho), np.float64)
    v = np.empty((3, N), np.float64)
    for a in range(3):
        v[a] = float(u[a])
    return r, v


def taylor_green(nx: int, ny: int, nz: int, u0: float, noise: float = 0.0, seed: int = 0,
                 two_d: bool = False):
    """Taylor-Green velocity field and density.  two_d drops the z dependence (cos(kz) -> 1)."""
    x, y, z = coords(nx, ny, nz)
    kx, ky, kz = 2 * math.pi / nx, 2 * math.pi / ny, 2 * math.pi / nz
    cz = np.ones_like(x, dtype=np.float64) if two_d else np.cos(kz * z)
    u = np.zeros((3, x.size), np.float64)
    u[0] = u0 * np.sin(kx * x) * np.cos(ky * y) * cz
    u[1] = -u0 * np.cos(kx * x) * np.sin(ky * y) * cz
    rho = np.ones(x.size, np.float64)
    if noise:
        rho += rng(seed).uniform(-noise, noise, size=x.size)
    return rho, u


def channel_flags(nx: int, ny: int, nz: int) -> np.ndarray:
    x, y, z = coords(nx, ny, nz)
    flags = np.zeros(x.size, np.uint8)
    flags[(y == 0) | (y == ny - 1)] = SOLID
    return flags


def sphere_flags(nx: int, ny: int, nz: int, center, radius: float,
                 inlet_x0: bool = True) -> np.ndarray:
    x, y, z = coords(nx, ny, nz)
    cx, cy, cz = center
    flags = np.zeros(x.size, np.uint8)
    inside = (x - cx) ** 2 + (y - cy) ** 2 + (z - cz) ** 2 <= radius * radius
    flags[inside] = SOLID
    if inlet_x0:
        flags[x == 0] = INLET
    return flags


def porous_flags(nx: int, ny: int, nz: int, solid_fraction: float = 0.30, blob: int = 3,
                 seed: int = SEED_POROUS512) -> np.ndarray:
    """Blobs of blob^3 cells at uniformly drawn lower corners, kept in draw order until the
    solid fraction first reaches `solid_fraction` (overlaps allowed, periodic wrap)."""
    N = nx * ny * nz
    target = int(math.ceil(solid_fraction * N))
    g = rng(seed)
    # first_cover[n]: index of the first blob (in draw order) that covers cell n
    first_cover = np.full(N, np.iinfo(np.int64).max, np.int64)
    drawn = 0
    batch = max(64, int(0.5 * N / blob ** 3))
    offsets = [(dx, dy, dz) for dz in range(blob) for dy in range(blob) for dx in range(blob)]
    while True:
        corner = g.integers(0, N, size=batch, dtype=np.int64)
        cx, cy, cz = corner % nx, (corner // nx) % ny, corner // (nx * ny)
        order = np.arange(drawn, drawn + batch, dtype=np.int64)
        for dx, dy, dz in offsets:
            cell = (cx + dx) % nx + nx * (((cy + dy) % ny) + ny * ((cz + dz) % nz))
            np.minimum.at(first_cover, cell, order)
        drawn += batch
        if int(np.count_nonzero(first_cover < drawn)) >= target:
            break
    # the smallest blob count K whose union reaches the target
    K = int(np.partition(first_cover, target - 1)[target - 1]) + 1
    flags = np.zeros(N, np.uint8)
    flags[first_cover < K] = SOLID
    return flags


def cavity_flags(nx: int, ny: int, nz: int) -> np.ndarray:
    """Lid-driven cavity: resting walls on the x, z and lower y faces, a MOVING_WALL lid on the
    layer y = ny - 1 (it covers the lid's edges)."""
    x, y, z = coords(nx, ny, nz)
    flags = np.zeros(x.size, np.uint8)
    flags[(x == 0) | (x == nx - 1) | (y == 0) | (z == 0) | (z == nz - 1)] = SOLID
    flags[y == ny - 1] = MOVING_WALL
    return flags


def labels(N: int) -> np.ndarray:
    """Distinct integer labels f[q, n] = 19 n + q + 1 (exact in fp32 while 19 N + 19 < 2^24)."""
    q = np.arange(19, dtype=np.int64)[:, None]
    n = np.arange(N, dtype=np.int64)[None, :]
    return (19 * n + q + 1).astype(np.float64)
