"""Domain decomposition of the lattice into z slabs, one per rank ("Disaggregated Design for
GPU-Based Volumetric Data Structures", section "Improving LBM Scalability": 1D partitioning along
one axis, each partition exchanging its boundary data with its two neighbours every time step).

Rank r of W owns the planes [z0, z1) of the global nz (a balanced split).  Its context holds
those planes plus one ghost plane below and one above (nz_local = z1 - z0 + 2): copies of the
neighbours' boundary planes, refreshed after every step.  The global z faces are periodic: the
neighbour below rank 0 is rank W - 1.  With W = 1 the slab exchanges with itself.

Per step: the engine steps its slab once, packs what its neighbours need from its first and last
owned planes (`lo` goes down, `hi` goes up), the ranks swap those buffers, and the engine
unpacks what it received into its ghost planes.  With the CUDA library (`LibraryEngine`) the
buffers are the five post-collision populations with c_z = -1 (lo) and c_z = +1 (hi) of the
boundary planes, in the library's internal storage, exchanged between device buffers: 10 nx ny
values per slab and step.  The momentum-exchange force of the owned cells is summed over ranks
(three doubles, an all-reduce).

An engine with begin() / end() overlaps the exchange with the interior planes ([Disaggregated],
"Disaggregation on a Dense Domain", OCC): begin() steps the two boundary planes, packs their
halos and starts the interior planes; the ranks swap the halos while the interior computes;
end() completes the step and unpacks.  The runner uses that form unless told otherwise.

This module holds no lattice Boltzmann arithmetic: the step, the packing and the unpacking run in
the engine (for `LibraryEngine`, the library's CUDA kernels).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Slab:
    rank: int
    world: int
    z0: int      # first owned global plane
    z1: int      # one past the last owned global plane
    below: int   # rank owning plane z0 - 1 (periodic)
    above: int   # rank owning plane z1 (periodic)
    nz_global: int

    @property
    def owned(self) -> int:
        return self.z1 - self.z0

    @property
    def local_nz(self) -> int:
        """Planes of the rank's context: the owned ones and two ghost planes."""
        return self.owned + 2

    def global_planes(self):
        """Global z of each local plane 0 .. local_nz - 1 (the ghosts wrap periodically)."""
        return [(self.z0 - 1 + k) % self.nz_global for k in range(self.local_nz)]


def slab_of(nz: int, rank: int, world: int) -> Slab:
    """Balanced split of nz planes over `world` ranks; every rank owns at least one plane."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of {world}")
    if nz < world:
        raise ValueError(f"{nz} planes cannot be split over {world} ranks")
    z0 = rank * nz // world
    z1 = (rank + 1) * nz // world
    return Slab(rank=rank, world=world, z0=z0, z1=z1, below=(rank - 1) % world,
                above=(rank + 1) % world, nz_global=nz)


def local_slice(global_array: np.ndarray, slab: Slab, nx: int, ny: int) -> np.ndarray:
    """The rank's local copy (ghost planes included) of a global array whose last axis is the cell
    index n = x + nx (y + ny z): the planes slab.global_planes(), in order."""
    planes = global_array.reshape(global_array.shape[:-1] + (slab.nz_global, ny * nx))
    local = planes[..., slab.global_planes(), :]
    return np.ascontiguousarray(local.reshape(global_array.shape[:-1] + (-1,)))


def owned_part(local_array: np.ndarray, slab: Slab, nx: int, ny: int) -> np.ndarray:
    """The owned planes of a local array (ghost planes dropped), last axis the local cell index."""
    planes = local_array.reshape(local_array.shape[:-1] + (slab.local_nz, ny * nx))
    return planes[..., 1:1 + slab.owned, :].reshape(local_array.shape[:-1] + (-1,))


class SlabRunner:
    """Steps one rank's slab and keeps its ghost planes current.

    engine: step1() -> None; pack() -> (lo, hi) tensors; unpack(from_below, from_above);
            local_force() -> three floats (the owned cells' momentum exchange); halo_like() -> an
            empty tensor of a halo buffer's shape, dtype and device.
    dist:   torch.distributed (an initialised process group) or None for a single rank."""

    def __init__(self, engine, slab: Slab, dist=None, group=None, overlap: bool = True):
        self.engine = engine
        self.slab = slab
        self.dist = dist
        self.group = group
        self.overlap = (overlap and callable(getattr(engine, "begin", None))
                        and callable(getattr(engine, "end", None)))
        if slab.world > 1 and dist is None:
            raise ValueError("several ranks need torch.distributed")
        self.from_below = engine.halo_like()
        self.from_above = engine.halo_like()

    def exchange(self) -> None:
        lo, hi = self.engine.pack()
        self._swap(lo, hi)
        self.engine.unpack(self.from_below, self.from_above)

    def _swap(self, lo, hi) -> None:
        """from_below <- the hi of the slab below, from_above <- the lo of the slab above."""
        s = self.slab
        if s.world == 1:
            # periodic in z on one rank: the slab is its own neighbour on both sides
            self.from_below.copy_(hi)
            self.from_above.copy_(lo)
        else:
            # the same order on every rank: hi goes up / from_below comes from below first, then
            # lo goes down / from_above comes from above (with two ranks both go to the same peer,
            # matched by order)
            ops = [self.dist.P2POp(self.dist.isend, hi, s.above, self.group),
                   self.dist.P2POp(self.dist.irecv, self.from_below, s.below, self.group)]
            for r in self.dist.batch_isend_irecv(ops):
                r.wait()
            ops = [self.dist.P2POp(self.dist.isend, lo, s.below, self.group),
                   self.dist.P2POp(self.dist.irecv, self.from_above, s.above, self.group)]
            for r in self.dist.batch_isend_irecv(ops):
                r.wait()

    def step(self, n: int) -> None:
        for _ in range(int(n)):
            if self.overlap:
                lo, hi = self.engine.begin()
                self._swap(lo, hi)
                self.engine.end(self.from_below, self.from_above)
            else:
                self.engine.step1()
                self.exchange()

    def force(self):
        """Force on the solids of the whole domain: the owned cells' sums, added over ranks."""
        local = np.asarray(self.engine.local_force(), np.float64)
        if self.slab.world == 1:
            return local
        import torch
        t = torch.tensor(local, dtype=torch.float64)
        dev = getattr(self.from_below, "device", None)
        if dev is not None and dev.type == "cuda":
            t = t.to(dev)
        self.dist.all_reduce(t, group=self.group)
        return t.cpu().numpy()


class LibraryEngine:
    """One rank's slab on the CUDA library: a context of nx x ny x (owned + 2) cells in the A-B
    scheme with ghost planes (lbm_set_ghost_planes), stepped one step at a time.  The context is
    moved to torch's current stream, which the communication calls order themselves against."""

    def __init__(self, ctx: int):
        import torch
        from . import binding as B
        self.B = B
        self.ctx = ctx
        B.lbm_set_stream(ctx, torch.cuda.current_stream().cuda_stream)
        elems = B.lbm_halo_elements(ctx)
        dtype = torch.float16 if B.lbm_halo_element_bytes(ctx) == 2 else torch.float32
        self._lo = torch.empty(elems, dtype=dtype, device="cuda")
        self._hi = torch.empty(elems, dtype=dtype, device="cuda")

    def halo_like(self):
        import torch
        return torch.empty_like(self._lo)

    def step1(self) -> None:
        self.B.lbm_step(self.ctx, 1)

    def pack(self):
        # enqueued on torch's current stream: a send issued after this waits for it
        self.B.lbm_halo_pack(self.ctx, self._lo, self._hi)
        return self._lo, self._hi

    def unpack(self, from_below, from_above) -> None:
        self.B.lbm_halo_unpack(self.ctx, from_below, from_above)

    def begin(self):
        # the boundary planes and the pack on torch's current stream, the interior on the
        # library's side stream: a send issued after this waits for the pack only
        self.B.lbm_slab_step_begin(self.ctx, self._lo, self._hi)
        return self._lo, self._hi

    def end(self, from_below, from_above) -> None:
        self.B.lbm_slab_step_end(self.ctx, from_below, from_above)

    def local_force(self):
        return self.B.lbm_force_momentum_exchange(self.ctx)
