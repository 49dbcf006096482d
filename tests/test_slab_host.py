"""Host logic of the z-slab decomposition (lattice_boltzmann_cfd_d3q19_gb300/slab.py), no GPU:
the partition, the ghost-plane mapping, the halo message order between gloo ranks and the force
reduction.  Each rank steps its slab with the CPU oracle (an engine that exchanges the boundary
planes' natural populations before every step), and the slabs together must equal the oracle's
unsliced run bit for bit ("Disaggregated Design for GPU-Based Volumetric Data Structures",
"Improving LBM Scalability": each partition exchanges its boundary data with its neighbours every
step)."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

from lattice_boltzmann_cfd_d3q19_gb300 import slab as S
from lattice_boltzmann_cfd_d3q19_gb300 import workloads as wl


@pytest.mark.parametrize("nz, world", [(12, 2), (13, 3), (5, 5), (7, 1)])
def test_partition_covers_every_plane_once(nz, world):
    slabs = [S.slab_of(nz, r, world) for r in range(world)]
    assert slabs[0].z0 == 0 and slabs[-1].z1 == nz
    for a, b in zip(slabs, slabs[1:]):
        assert a.z1 == b.z0
    sizes = [s.owned for s in slabs]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    for s in slabs:
        assert slabs[s.below].z1 % nz == s.z0 and slabs[s.above].z0 == s.z1 % nz
        assert s.global_planes() == [(s.z0 - 1 + k) % nz for k in range(s.owned + 2)]


def test_partition_rejects_too_many_ranks():
    with pytest.raises(ValueError):
        S.slab_of(3, 0, 4)


def test_local_slice_and_owned_part_round_trip():
    nx, ny, nz = 3, 2, 7
    a = np.arange(2 * nx * ny * nz).reshape(2, -1)
    parts = []
    for r in range(3):
        s = S.slab_of(nz, r, 3)
        loc = S.local_slice(a, s, nx, ny)
        assert loc.shape == (2, nx * ny * s.local_nz)
        # ghost planes are the neighbours' boundary planes
        planes = loc.reshape(2, s.local_nz, nx * ny)
        glob = a.reshape(2, nz, nx * ny)
        assert np.array_equal(planes[:, 0], glob[:, (s.z0 - 1) % nz])
        assert np.array_equal(planes[:, -1], glob[:, s.z1 % nz])
        parts.append(S.owned_part(loc, s, nx, ny))
    assert np.array_equal(np.concatenate(parts, axis=1), a)


# ---- ranks stepping their slabs with the oracle ------------------------------------------------------

NX, NY, TAU, G, STEPS = 10, 8, 0.62, (2e-5, -1e-5, 1e-5), 5


def problem(nz):
    r = np.random.default_rng(4040)
    N = NX * NY * nz
    flags = (r.uniform(size=N) < 0.15).astype(np.uint8)
    x, _, _ = wl.coords(NX, NY, nz)
    flags[x == 0] = wl.INLET
    rho = 1 + r.uniform(-0.02, 0.02, N)
    u = r.uniform(-0.03, 0.03, (3, N))
    return flags, rho, u


class OracleEngine:
    """A slab stepped by the CPU oracle: its ghost planes hold the neighbours' boundary planes'
    natural populations (all 19), which is what the oracle's two-lattice step needs there."""

    def __init__(self, slab, f_local, flags_local):
        import oracle
        self.slab = slab
        self.P = oracle.Problem(NX, NY, slab.local_nz, TAU, flags=flags_local, faces=(1, 0, 0),
                                inlet=(1.0, 0.04, 0.0, 0.0), g=G)
        self.f = f_local.copy()
        self.area = NX * NY

    def _plane(self, k):
        return self.f.reshape(19, self.slab.local_nz, self.area)[:, k]

    def halo_like(self):
        import torch
        return torch.empty(19 * self.area, dtype=torch.float64)

    def step1(self):
        self.f, _ = self.P.step_ab(self.f, 1)

    def pack(self):
        import torch
        lo = torch.from_numpy(np.ascontiguousarray(self._plane(1)).reshape(-1))
        hi = torch.from_numpy(np.ascontiguousarray(self._plane(self.slab.local_nz - 2)).reshape(-1))
        return lo, hi

    def unpack(self, from_below, from_above):
        planes = self.f.reshape(19, self.slab.local_nz, self.area)
        planes[:, 0] = from_below.numpy().reshape(19, self.area)
        planes[:, -1] = from_above.numpy().reshape(19, self.area)

    def local_force(self):
        # a per-rank value whose sum over ranks is known: checks the reduction only
        return (float(self.slab.rank + 1), 0.5, -float(self.slab.z0))

    # the overlapped form: the oracle has no interior to run beside the exchange, so begin() is
    # the whole step and the pack, end() the unpack; what this checks is the runner's order
    def begin(self):
        self.step1()
        return self.pack()

    def end(self, from_below, from_above):
        self.unpack(from_below, from_above)


class SerialOracleEngine(OracleEngine):
    begin = None
    end = None


def _rank_main(rank, world, nz, port, out, overlap=True):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        flags, rho, u = problem(nz)
        f0 = oracle.equilibrium_field(rho, u)
        s = S.slab_of(nz, rank, world)
        cls = OracleEngine if overlap else SerialOracleEngine
        eng = cls(s, S.local_slice(f0, s, NX, NY), S.local_slice(flags, s, NX, NY))
        run = S.SlabRunner(eng, s, dist)
        assert run.overlap == overlap
        run.step(STEPS)
        F = run.force()
        out.put((rank, S.owned_part(eng.f, s, NX, NY), F))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("nz, world", [(12, 2), (13, 3)])
def test_slabs_on_gloo_ranks_equal_the_unsliced_oracle(nz, world, overlap):
    import oracle
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, nz, port, q, overlap))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (f, F)) for r, f, F in (q.get(timeout=300) for _ in procs))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    flags, rho, u = problem(nz)
    P = oracle.Problem(NX, NY, nz, TAU, flags=flags, faces=(1, 0, 0), inlet=(1.0, 0.04, 0.0, 0.0),
                       g=G)
    ref, _ = P.step_ab(oracle.equilibrium_field(rho, u), STEPS)
    got = np.concatenate([res[r][0] for r in range(world)], axis=1)
    fluid = flags == wl.FLUID
    assert np.array_equal(got[:, fluid], ref[:, fluid])
    # the force is the sum of the ranks' owned-cell sums, the same on every rank
    want = np.array([sum(r + 1 for r in range(world)), 0.5 * world,
                     -sum(S.slab_of(nz, r, world).z0 for r in range(world))])
    for r in range(world):
        assert np.allclose(res[r][1], want)
