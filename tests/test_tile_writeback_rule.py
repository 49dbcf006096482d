"""The write-back rule of the collision layout's tiled AA odd step on grids without solid links,
checked on the CPU by brute force.

In the AA odd step population q of cell x goes to element q of the record of x + c_q, so element
q of the record of r has the one writer r - c_q.  A block of the tiled kernel holds a tile of
32 x t_y cells of a chunk of t_z planes plus a one-cell halo; without solid links it writes back
the elements whose writer lies in its tile and chunk, taken per axis: a record at position p of a
span of t cells (p = -1 and p = t the halo) takes the elements whose velocity component c has
p - c in [0, t - 1].  Here that rule is compared with the elements every cell of an all-fluid
block actually writes, on the tile shapes the kernel meets (ragged last rows, chunks of one plane,
a single chunk), together with the list of the 160 records of a plane inside the chunk that do not
go back whole, and the shared-memory offsets the write-back reads."""
import itertools

# D3Q19 velocities (the order does not matter here: only the set of components does)
VEL = [c for c in itertools.product((-1, 0, 1), repeat=3) if sum(map(abs, c)) <= 2]
TX, TY = 32, 8
HX, HY = TX + 2, TY + 2
ROW_FLOATS = 648            # a halo row in shared memory: a pad float, 34 records, padding
PLANE_FLOATS = HY * ROW_FLOATS


def vel_mask(axis, c):
    return sum(1 << q for q, v in enumerate(VEL) if v[axis] == c)


def axis_mask(axis, pos, t):
    return ((vel_mask(axis, -1) if -1 <= pos <= t - 2 else 0)
            | (vel_mask(axis, 0) if 0 <= pos <= t - 1 else 0)
            | (vel_mask(axis, 1) if 1 <= pos <= t else 0))


def whole_record(rid, ty_n):
    hx, hy = rid % HX, rid // HX
    return 2 <= hx <= TX - 1 and 2 <= hy <= TY - 1 and hy < ty_n


def edge_record(c):
    """The c-th record of a plane inside the chunk that does not go back whole (full tiles)."""
    if c < 2 * HX:
        return (0 if c < HX else (HY - 1) * HX) + c % HX
    if c < 2 * HX + 4 * (TY - 2):
        i = c - 2 * HX
        k = i & 3
        return (2 + (i >> 2)) * HX + (k if k < 2 else TX - 2 + k)
    i = c - 2 * HX - 4 * (TY - 2)
    return (1 if i < HX else TY) * HX + i % HX


def test_velocity_set():
    assert len(VEL) == 19 and (0, 0, 0) in VEL
    assert all(bin(vel_mask(a, -1)).count("1") == 5 for a in range(3))


def test_rule_equals_the_elements_an_all_fluid_block_writes():
    # (rows of the tile inside the grid, planes of the chunk)
    for ty_n, t_z in itertools.product(range(1, TY + 1), (1, 2, 3, 7, 15)):
        written = {}
        for z, ty, tx in itertools.product(range(t_z), range(ty_n), range(TX)):
            for q, (cx, cy, cz) in enumerate(VEL):
                key = (z + cz, (ty + 1 + cy) * HX + (tx + 1 + cx))  # (plane, halo record)
                written[key] = written.get(key, 0) | (1 << q)
        rule = {}
        for pz in range(-1, t_z + 1):
            mz = axis_mask(2, pz, t_z)
            for rid in range(HX * HY):
                m = axis_mask(0, rid % HX - 1, TX) & axis_mask(1, rid // HX - 1, ty_n) & mz
                if m:
                    rule[(pz, rid)] = m
        assert rule == written, (ty_n, t_z)


def test_whole_records_and_the_edge_list_cover_a_plane_inside_the_chunk():
    edge = [edge_record(c) for c in range(160)]
    assert len(set(edge)) == 160
    assert set(edge) == {r for r in range(HX * HY) if not whole_record(r, TY)}
    # a record that goes back whole is written in all 19 elements by the block's own cells
    full = (1 << 19) - 1
    for r in range(HX * HY):
        m = axis_mask(0, r % HX - 1, TX) & axis_mask(1, r // HX - 1, TY)
        assert (m == full) == whole_record(r, TY), r
    # the edge rows' records (14 elements) go to the warps that hold no whole row
    heavy = [c for c in range(160) if bin(axis_mask(0, edge[c] % HX - 1, TX)
                                         & axis_mask(1, edge[c] // HX - 1, TY)).count("1") == 14]
    warps = {(96 + c) // 32 for c in heavy}
    assert warps <= {5, 6, 7}, warps


def test_shared_memory_offsets_stay_in_the_plane():
    last = max(hy * ROW_FLOATS + 1 + hx * 19 + 18 for hx in range(HX) for hy in range(HY))
    assert last < PLANE_FLOATS
