// The A-B pull in the collision layout with its gather staged through shared memory in 2.5D
// blocks.  In that layout a cell's 19 populations form one 76-byte record ([PortLBM] §3.2,
// Fig. 2(b)), and the pull reads element q of the record of x - c_q.  Element by element, a warp's
// request touches a sector per lane, and each source record's sectors are fetched from the L2
// once for every cell that needs one of its elements (about 615 bytes per cell at 256^3, for the
// 76 the cell needs).  Here a block holds whole records of its x-y tile plus a one-cell halo for
// three z planes, copied in coalesced runs, and walks its tile along z: every record crosses the
// L2 about (10 x 34) / (8 x 32) times per plane.
#pragma once

#include "lbm_kernels.cuh"

namespace lbm {

// kTileX (32: one warp per row) by kTileY rows: lbm_device.cuh
constexpr int kTileThreads = kTileX * kTileY;
constexpr int kHaloX = kTileX + 2;
constexpr int kHaloY = kTileY + 2;
// A halo row in shared memory: one pad float, then the records of x0 - 1 .. x0 + 32 in order
// (hx = 0 .. 33 at 1 + 19 hx), so that the run x0 .. x0 + 31 starts at float 20, 16-byte aligned
// like its source (76 (row + x0) bytes with 32 | nx), and the row is padded to 648 floats.
constexpr int kTileRowFloats = 648;
constexpr int kTileRunFloats = kTileX * 19;                  // 608: one row's own records
constexpr int kTileRunPieces = kTileRunFloats / 4;           // 152 pieces of 16 bytes
constexpr int kTilePlaneFloats = kHaloY * kTileRowFloats;    // one plane of the ring
static_assert(1 + kHaloX * 19 <= kTileRowFloats && kTileRowFloats % 4 == 0, "halo row layout");
constexpr int kTileSlots = 4;  // planes z - 1, z, z + 1 being read, z + 2 arriving
constexpr size_t kTileSmemBytes = kTileSlots * kTilePlaneFloats * sizeof(float);
static_assert(kTileY * kTileX * 19 <= kTilePlaneFloats, "a tile's results fit in one slot");

// coordinate v in [-1, n] of a source row: wrapped on a PERIODIC axis, clamped onto the last
// layer on an OPEN one (the zero-gradient source of a pull); v > n only for rows of the ragged
// tail that no cell reads, kept in range
__device__ __forceinline__ int tile_edge(int v, int n, bool open) {
    if (v < 0) return open ? 0 : n - 1;
    if (v == n) return open ? n - 1 : 0;
    return v < n ? v : n - 1;
}

__device__ __forceinline__ void cp_async4(float* dst_shared, const float* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst_shared);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst_shared, const float* src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst_shared);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most `pending` of this thread's committed groups are still in flight
template <int pending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(pending) : "memory"); }

__device__ __forceinline__ int tile_slot(int z) { return (z + kTileSlots) % kTileSlots; }  // z >= -1

// Plane zs of A, rows y0 - 1 .. y0 + kTileY, into `dst` (kHaloY halo rows).  In every row thread
// t < 152 copies the 16-byte piece t of the run x0 .. x0 + 31.  The edge records x0 - 1 and
// x0 + 32 follow.  Where such a record is the run's neighbour in memory, it is one aligned block
// of 80 bytes (5 pieces; the extra float lands on a pad float of the halo row, and with 32 | nx the
// block never leaves the row).  Where it is wrapped or clamped, it is 19 single elements.
// Asynchronous; the caller commits the group.
// clamp: OPEN axes clamp onto the last layer (the A-B pull); otherwise every axis wraps (the AA
// odd step, whose links across an OPEN face belong to special cells).
__device__ __forceinline__ void tile_load_plane(const Params& p, const float* A, float* dst, int x0,
                                                int y0, int zs, bool clamp = true) {
    const int t = (int)threadIdx.x;
    const bool lw = x0 > 0, rw = x0 + kTileX < p.nx;
    const int nl = lw ? 5 : 19, nr = rw ? 5 : 19;
    bool wide;
    uint32_t src;  // element offset from the row's first element
    int d;         // float offset in the halo row
    if (t < kTileRunPieces) {
        wide = true;
        src = 19u * (uint32_t)x0 + 4u * (uint32_t)t;
        d = 20 + 4 * t;
    } else if (t < kTileRunPieces + nl) {
        const int i = t - kTileRunPieces;
        wide = lw;
        if (lw) {
            src = 19u * (uint32_t)x0 - 20u + 4u * (uint32_t)i;
            d = 4 * i;
        } else {
            src = 19u * (uint32_t)tile_edge(x0 - 1, p.nx, clamp && p.open[0]) + (uint32_t)i;
            d = 1 + i;
        }
    } else if (t < kTileRunPieces + nl + nr) {
        const int i = t - kTileRunPieces - nl;
        wide = rw;
        if (rw) {
            src = 19u * (uint32_t)(x0 + kTileX) + 4u * (uint32_t)i;
            d = 1 + (kHaloX - 1) * 19 + 4 * i;
        } else {
            src = 19u * (uint32_t)tile_edge(x0 + kTileX, p.nx, clamp && p.open[0]) + (uint32_t)i;
            d = 1 + (kHaloX - 1) * 19 + i;
        }
    } else {
        return;
    }
#pragma unroll 2
    for (int r = 0; r < kHaloY; ++r) {
        const int y = tile_edge(y0 - 1 + r, p.ny, clamp && p.open[1]);
        const uint32_t row = (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * (uint32_t)zs);
        const float* g = A + (19u * row + src);
        float* s_ = dst + r * kTileRowFloats + d;
        if (wide) cp_async16(s_, g);
        else cp_async4(s_, g);
    }
}

// population q of the cell at (tx, ty) of the tile from the ring: element q of the record of
// x - c_q, or on a solid link opposite(q) element opposite(q) of its own record
template <int Q = 0>
__device__ __forceinline__ void tile_gather(const float* pm, const float* p0, const float* pp,
                                            int own, uint32_t m, float (&h)[19]) {
    constexpr int dz = cz(Q);
    const float* src = dz > 0 ? pm : dz < 0 ? pp : p0;
    const int off = own - cy(Q) * kTileRowFloats - cx(Q) * 19;
    if constexpr (Q == 0) h[Q] = src[off + Q];
    else h[Q] = solid_link<opp(Q)>(m) ? p0[own + opp(Q)] : src[off + Q];
    if constexpr (Q < 18) tile_gather<Q + 1>(pm, p0, pp, own, m, h);
}

// Grid: (nx / 32, ceil(ny / 8), chunks); a block walks the planes of its chunk of
// ceil(nz / chunks).  FLUID cells that are not special are pulled and collided; INLET cells store
// the reservoir's f_eq, the others zeros (the boundary kernel, launched after this one, writes the
// special cells).  The caller checks 32 | nx and 19 N <= 2^32.
// Pipeline: while plane z is computed from the slots of z - 1, z and z + 1, the copies of z + 2
// are in flight; after it, the results go through the freed slot of z - 1 to the destination in
// one run per row, and the copies of z + 3 start into that slot.
// WALLS = false: the grid has no solid link (masks known zero, the bounce-back selects fold away)
template <bool FORCE, bool BODY, bool WALLS = true>
__global__ void __launch_bounds__(kTileThreads, 2) k_ab_pull_tile(Params p) {
    extern __shared__ __align__(16) float tile_smem[];
    float* ring = tile_smem;
    const int tx = (int)threadIdx.x & 31, ty = (int)threadIdx.x >> 5;
    const int x0 = (int)blockIdx.x * kTileX, y0 = (int)blockIdx.y * kTileY;
    const int len = (p.nz + (int)gridDim.z - 1) / (int)gridDim.z;
    const int z0 = (int)blockIdx.z * len;
    const int z1 = min(z0 + len, p.nz);
    const int x = x0 + tx, y = y0 + ty;
    const bool row_in = y < p.ny;  // the same for the whole warp
    const float* A = static_cast<const float*>(p.A);
    float* B = static_cast<float*>(p.B);
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (z0 < z1) {
        // planes z0 - 1 .. z0 + 1 (one group), then z0 + 2 (the next); a plane is needed up to z1
        for (int z = z0 - 1; z <= z0 + 1; ++z)
            tile_load_plane(p, A, ring + tile_slot(z) * kTilePlaneFloats, x0, y0,
                            tile_edge(z, p.nz, p.open[2]));
        cp_async_commit();
        if (z0 + 2 <= z1)
            tile_load_plane(p, A, ring + tile_slot(z0 + 2) * kTilePlaneFloats, x0, y0,
                            tile_edge(z0 + 2, p.nz, p.open[2]));
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int own = (ty + 1) * kTileRowFloats + 1 + (tx + 1) * 19;
        const uint32_t area = (uint32_t)p.nx * (uint32_t)p.ny;
        uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * (uint32_t)z0);
        // the flag byte and mask of a cell are loaded one plane ahead of its use
        uint32_t m_next = 0u;
        uint8_t fl_next = (uint8_t)T_SOLID;
        if (row_in) {
            m_next = (WALLS && p.any_solid_link) ? p.mask[n] : 0u;
            fl_next = p.flags[n];
        }
        for (int z = z0; z < z1; ++z, n += area) {
            float h[19];
            const uint32_t m = m_next;
            const uint8_t fl = fl_next;
            if (row_in && z + 1 < z1) {
                m_next = (WALLS && p.any_solid_link) ? p.mask[n + area] : 0u;
                fl_next = p.flags[n + area];
            }
            if (row_in) {
                if ((fl & (TYPE_MASK | F_SPECIAL)) == T_FLUID) {
                    tile_gather(ring + tile_slot(z - 1) * kTilePlaneFloats,
                                ring + tile_slot(z) * kTilePlaneFloats,
                                ring + tile_slot(z + 1) * kTilePlaneFloats, own, m, h);
                    collide<BODY>(h, p);
                    if (FORCE && m) mask_forces(m, h, fx, fy, fz);
                } else {
                    const bool inl = p.any_inlet && (fl & TYPE_MASK) == T_INLET;
#pragma unroll
                    for (int q = 0; q < 19; ++q) h[q] = inl ? p.heq_in[q] : 0.0f;
                }
            }
            __syncthreads();  // every read of the slot of z - 1 is done
            float* out = ring + tile_slot(z - 1) * kTilePlaneFloats;
            if (row_in) {
                float* o = out + ty * kTileRunFloats + tx * 19;
#pragma unroll
                for (int q = 0; q < 19; ++q) o[q] = h[q];
            }
            __syncwarp();
            if (row_in) {
                // the row's 32 records are one contiguous, 16-byte aligned run of the destination
                float4* dst = reinterpret_cast<float4*>(B + 19u * (n - (uint32_t)tx));
                const float4* src = reinterpret_cast<const float4*>(out + ty * kTileRunFloats);
                for (int k = tx; k < kTileRunPieces; k += 32) dst[k] = src[k];
            }
            __syncthreads();  // the slot of z - 1 is free again
            if (z + 3 <= z1)
                tile_load_plane(p, A, ring + tile_slot(z + 3) * kTilePlaneFloats, x0, y0,
                                tile_edge(z + 3, p.nz, p.open[2]));
            cp_async_commit();
            cp_async_wait<1>();  // plane z + 2 has arrived (z + 3 may still be in flight)
            __syncthreads();
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

// ============================== AA odd step, collision layout, 2.5D tiles ========================
// The AA odd step writes population q of cell x into element q of the record of x + c_q, so in the
// collision layout a record's elements come from 19 cells and every element store of a warp hit
// another sector: each sector was assembled in the L2 from about eight 4-byte writes.  Here a block
// updates the records of its tile and halo in place in shared memory.  Each cell reads and writes
// only its own slot set (the AA property), plus, on a solid link, one slot of its own record that
// the SOLID neighbour owns and nobody else writes.  A plane is final once the plane after it has
// been computed, and then it goes back to the buffer.
// * Records whose 19 slots all belong to this block's cells go back whole, one contiguous run per
//   row: x-y interior records (hx 2 .. 31, hy 2 .. 7 with the next row inside the grid) of planes
//   strictly inside the block's chunk.
// * Every other record goes back element by element: only the slots this block wrote, recorded
//   in a 32-bit mask per record.  On a grid without solid links the slots follow from geometry
//   (each has one writer, x - c_q) and no mask is kept: the write-back takes them per axis, and the
//   160 such records of a plane inside the chunk go one to a thread.
// The whole records carry stale values in the slots of special cells, so the boundary kernel runs
// after this kernel, not beside it.  The caller checks 32 | nx, ny >= kTileY + 2 (no two rows of a
// halo tile are the same row of the grid) and 19 N <= 2^32.
constexpr int kTileRecords = kHaloX * kHaloY;
constexpr size_t kOddTileSmemBytes = kTileSmemBytes + kTileSlots * kTileRecords * sizeof(uint32_t);

// v in [-n, 2 n): the halo coordinates of a tile (x in [-1, nx], y in [-1, ny + 8] with ny >= 10,
// z in [-1, nz])
__device__ __forceinline__ int tile_wrap(int v, int n) { return v < 0 ? v + n : v >= n ? v - n : v; }

// population q of the cell from element opposite(q) of the record of x - c_q, or on a solid link
// opposite(q) element q of its own record (the AA odd gather)
template <int Q = 0>
__device__ __forceinline__ void tile_odd_gather(const float* pm, const float* p0, const float* pp,
                                                int own, uint32_t m, float (&h)[19]) {
    constexpr int dz = cz(Q);
    const float* src = dz > 0 ? pm : dz < 0 ? pp : p0;
    constexpr int shift = -cy(Q) * kTileRowFloats - cx(Q) * 19 + opp(Q);
    if constexpr (Q == 0) h[Q] = p0[own];
    else h[Q] = solid_link<opp(Q)>(m) ? p0[own + Q] : src[own + shift];
    if constexpr (Q < 18) tile_odd_gather<Q + 1>(pm, p0, pp, own, m, h);
}

// population q to element q of the record of x + c_q, or on a solid link q to element opposite(q)
// of its own record (with the link's momentum exchange); BITS: the element's bit is set in its
// record's mask (on a grid without solid links the elements written follow from geometry instead)
template <bool FORCE, bool BITS, int Q = 0>
__device__ __forceinline__ void tile_odd_scatter(float* pm, float* p0, float* pp, uint32_t* bm,
                                                 uint32_t* b0, uint32_t* bp, int own, int rid,
                                                 uint32_t m, const float (&h)[19], float& fx,
                                                 float& fy, float& fz) {
    constexpr int dz = cz(Q);
    if (Q > 0 && solid_link<Q>(m)) {
        p0[own + opp(Q)] = h[Q];
        if (BITS) atomicOr(&b0[rid], 1u << opp(Q));
        if (FORCE) accumulate_force<Q>(h[Q], fx, fy, fz);
    } else {
        float* dst = dz > 0 ? pp : dz < 0 ? pm : p0;
        dst[own + cy(Q) * kTileRowFloats + cx(Q) * 19 + Q] = h[Q];
        if (BITS) {
            uint32_t* bd = dz > 0 ? bp : dz < 0 ? bm : b0;
            atomicOr(&bd[rid + cy(Q) * kHaloX + cx(Q)], 1u << Q);
        }
    }
    if constexpr (Q < 18)
        tile_odd_scatter<FORCE, BITS, Q + 1>(pm, p0, pp, bm, b0, bp, own, rid, m, h, fx, fy, fz);
}

// INLET producer: f_eq,q of the reservoir to element q of the record of s + c_q, links that leave
// the grid through an OPEN face dropped (as the one-cell kernel's producer)
template <bool BITS, int Q = 1>
__device__ __forceinline__ void tile_odd_produce(const Params& p, float* pm, float* p0, float* pp,
                                                 uint32_t* bm, uint32_t* b0, uint32_t* bp, int own,
                                                 int rid, int x, int y, int z) {
    if (!leaves_open(p, x, y, z, cx(Q), cy(Q), cz(Q))) {
        constexpr int dz = cz(Q);
        float* dst = dz > 0 ? pp : dz < 0 ? pm : p0;
        dst[own + cy(Q) * kTileRowFloats + cx(Q) * 19 + Q] = p.heq_in[Q];
        if (BITS) {
            uint32_t* bd = dz > 0 ? bp : dz < 0 ? bm : b0;
            atomicOr(&bd[rid + cy(Q) * kHaloX + cx(Q)], 1u << Q);
        }
    }
    if constexpr (Q < 18) tile_odd_produce<BITS, Q + 1>(p, pm, p0, pp, bm, b0, bp, own, rid, x, y, z);
}

// the elements of mask b of record rid of the ring's plane `ring_s` to plane gz of A
__device__ __forceinline__ void tile_odd_put(const Params& p, float* A, const float* ring_s, int x0,
                                             int y0, uint32_t gz, int rid, uint32_t b) {
    const int hx = rid % kHaloX, hy = rid / kHaloX;
    const uint32_t gx = (uint32_t)tile_wrap(x0 - 1 + hx, p.nx);
    const uint32_t gy = (uint32_t)tile_wrap(y0 - 1 + hy, p.ny);
    float* dst = A + 19u * (gx + (uint32_t)p.nx * (gy + (uint32_t)p.ny * gz));
    const float* src = ring_s + hy * kTileRowFloats + 1 + hx * 19;
    for (uint32_t r = b; r; r &= r - 1u) {
        const int e = __ffs(r) - 1;
        dst[e] = src[e];
    }
}

// `whole`: the x-y interior records of plane gz (hx 2 .. 31, hy 2 .. 7 with the next row inside
// the grid) back to A in contiguous runs, warp w taking row hy = 2 + w (30 records)
__device__ __forceinline__ void tile_odd_put_whole(const Params& p, float* A, const float* ring_s,
                                                   int x0, int y0, uint32_t gz) {
    const int t = (int)threadIdx.x;
    const int w = t >> 5, lane = t & 31;
    const int hy = 2 + w;
    if (w < kTileY - 2 && y0 + hy < p.ny) {
        const uint32_t gy = (uint32_t)(y0 + hy - 1);
        float* dst = A + 19u * ((uint32_t)(x0 + 1) + (uint32_t)p.nx * (gy + (uint32_t)p.ny * gz));
        const float* src = ring_s + hy * kTileRowFloats + 1 + 2 * 19;
        for (int k = lane; k < (kTileX - 2) * 19; k += 32) dst[k] = src[k];
    }
}
__device__ __forceinline__ bool tile_whole_record(int rid, int y0, int ny) {
    const int hx = rid % kHaloX, hy = rid / kHaloX;
    return hx >= 2 && hx <= kTileX - 1 && hy >= 2 && hy <= kTileY - 1 && y0 + hy < ny;
}

// plane pl of the ring (slot `ring_s`, masks `bits_s`) back to A; `whole`: the plane lies
// strictly inside the chunk, so its x-y interior records go back whole.  The masks are cleared.
__device__ __forceinline__ void tile_odd_writeback(const Params& p, float* A, const float* ring_s,
                                                   uint32_t* bits_s, int x0, int y0, int pl,
                                                   bool whole) {
    const uint32_t gz = (uint32_t)tile_wrap(pl, p.nz);
    if (whole) tile_odd_put_whole(p, A, ring_s, x0, y0, gz);
    for (int rid = (int)threadIdx.x; rid < kTileRecords; rid += kTileThreads) {
        const uint32_t b = bits_s[rid];
        if (b == 0u) continue;
        bits_s[rid] = 0u;
        if (whole && tile_whole_record(rid, y0, p.ny)) continue;
        tile_odd_put(p, A, ring_s, x0, y0, gz, rid, b);
    }
}

// On a grid without solid links every element of the AA odd step has one writer by geometry:
// element q of the record of x is written by the cell x - c_q, whatever that cell's type (a cell
// that is not updated leaves the value loaded with the plane, which goes back unchanged; the
// special cells' boundary kernel runs after this kernel).  So the elements a block writes back
// are those whose writer lies in its tile and chunk, with no per-element record: along one axis,
// a record at position p of a span of t cells (p = -1 and p = t its halo) takes the elements
// whose c along the axis has p - c in [0, t - 1].
constexpr uint32_t tile_vel_mask(int axis, int c) {
    uint32_t m = 0u;
    for (int q = 0; q < 19; ++q)
        if ((axis == 0 ? cx(q) : axis == 1 ? cy(q) : cz(q)) == c) m |= 1u << q;
    return m;
}
template <int AXIS>
__device__ __forceinline__ uint32_t tile_axis_mask(int pos, int t) {
    constexpr uint32_t lo = tile_vel_mask(AXIS, -1), mid = tile_vel_mask(AXIS, 0),
                       hi = tile_vel_mask(AXIS, 1);
    return (pos >= -1 && pos <= t - 2 ? lo : 0u) | (pos >= 0 && pos <= t - 1 ? mid : 0u) |
           (pos >= 1 && pos <= t ? hi : 0u);
}
__device__ __forceinline__ uint32_t tile_xy_mask(int rid, int ty_n) {
    const int hx = rid % kHaloX, hy = rid / kHaloX;
    return tile_axis_mask<0>(hx - 1, kTileX) & tile_axis_mask<1>(hy - 1, ty_n);
}
// The records of a plane that do not go back whole, when all kTileY rows of the tile are in the
// grid: halo rows hy = 0 and 9 (c 0 .. 67), the columns hx = 0, 1, 32, 33 of rows 2 .. 7
// (c 68 .. 91), edge rows hy = 1 and 8 (c 92 .. 159); given to threads 96 .. 255, so that warps 6
// and 7, which hold no whole row, take the edge rows, whose records have 14 elements each.
constexpr int kTileEdgeRecords = 4 * kHaloX + 4 * (kTileY - 2);
static_assert(kTileEdgeRecords == 160 && kTileThreads - 96 == kTileEdgeRecords, "edge record list");
__device__ __forceinline__ int tile_edge_record(int c) {
    if (c < 2 * kHaloX) return (c < kHaloX ? 0 : (kHaloY - 1) * kHaloX) + c % kHaloX;
    if (c < 2 * kHaloX + 4 * (kTileY - 2)) {
        const int i = c - 2 * kHaloX, k = i & 3;
        return (2 + (i >> 2)) * kHaloX + (k < 2 ? k : kTileX - 2 + k);
    }
    const int i = c - 2 * kHaloX - 4 * (kTileY - 2);
    return (i < kHaloX ? 1 : kTileY) * kHaloX + i % kHaloX;
}
// A thread's records of the static write-back and their x-y masks: rid = t and t + 256 of a plane
// written record by record, and its record of the list above (thread t >= 96, full tiles)
struct TileOwned {
    uint32_t m0 = 0u, m1 = 0u, me = 0u;
    int re = 0;
    __device__ __forceinline__ TileOwned(int y0, int ny) {
        const int t = (int)threadIdx.x;
        const int ty_n = min(kTileY, ny - y0);
        m0 = tile_xy_mask(t, ty_n);
        if (t + kTileThreads < kTileRecords) m1 = tile_xy_mask(t + kTileThreads, ty_n);
        if (t >= kTileThreads - kTileEdgeRecords && ty_n == kTileY) {
            re = tile_edge_record(t - (kTileThreads - kTileEdgeRecords));
            me = tile_xy_mask(re, ty_n);
        }
    }
};
// plane pl of the ring back to A on a grid without solid links; mz: the plane's z mask
__device__ __forceinline__ void tile_odd_writeback_static(const Params& p, float* A,
                                                          const float* ring_s, int x0, int y0,
                                                          int pl, uint32_t mz, bool whole,
                                                          const TileOwned& o) {
    const uint32_t gz = (uint32_t)tile_wrap(pl, p.nz);
    const int t = (int)threadIdx.x;
    if (whole) {
        tile_odd_put_whole(p, A, ring_s, x0, y0, gz);
        if (y0 + kTileY <= p.ny) {
            if (o.me) tile_odd_put(p, A, ring_s, x0, y0, gz, o.re, o.me);
            return;
        }
    }
    if (const uint32_t b = o.m0 & mz; b && !(whole && tile_whole_record(t, y0, p.ny)))
        tile_odd_put(p, A, ring_s, x0, y0, gz, t, b);
    if (const uint32_t b = o.m1 & mz; b && !(whole && tile_whole_record(t + kTileThreads, y0, p.ny)))
        tile_odd_put(p, A, ring_s, x0, y0, gz, t + kTileThreads, b);
}

// Grid: (nx / 32, ceil(ny / 8), chunks), as the tiled pull.  FLUID cells that are not special are
// gathered, collided and scattered; INLET cells produce.
template <bool FORCE, bool BODY, bool WALLS = true>
__global__ void __launch_bounds__(kTileThreads, 2) k_aa_odd_tile(Params p) {
    extern __shared__ __align__(16) float tile_smem[];
    float* ring = tile_smem;
    uint32_t* bits = reinterpret_cast<uint32_t*>(tile_smem + kTileSlots * kTilePlaneFloats);
    const int tx = (int)threadIdx.x & 31, ty = (int)threadIdx.x >> 5;
    const int x0 = (int)blockIdx.x * kTileX, y0 = (int)blockIdx.y * kTileY;
    const int len = (p.nz + (int)gridDim.z - 1) / (int)gridDim.z;
    const int z0 = (int)blockIdx.z * len;
    const int z1 = min(z0 + len, p.nz);
    const int x = x0 + tx, y = y0 + ty;
    const bool row_in = y < p.ny;  // the same for the whole warp
    float* A = static_cast<float*>(p.A);
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (z0 < z1) {
        if (WALLS)
            for (int k = (int)threadIdx.x; k < kTileSlots * kTileRecords; k += kTileThreads) bits[k] = 0u;
        const TileOwned owned(y0, p.ny);  // the geometric write-back (grids without solid links)
        for (int z = z0 - 1; z <= z0 + 1; ++z)
            tile_load_plane(p, A, ring + tile_slot(z) * kTilePlaneFloats, x0, y0,
                            tile_wrap(z, p.nz), false);
        cp_async_commit();
        if (z0 + 2 <= z1)
            tile_load_plane(p, A, ring + tile_slot(z0 + 2) * kTilePlaneFloats, x0, y0,
                            tile_wrap(z0 + 2, p.nz), false);
        cp_async_commit();
        const int own = (ty + 1) * kTileRowFloats + 1 + (tx + 1) * 19;
        const int rid = (ty + 1) * kHaloX + (tx + 1);
        const uint32_t area = (uint32_t)p.nx * (uint32_t)p.ny;
        uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * (uint32_t)z0);
        uint32_t m_next = 0u;
        uint8_t fl_next = (uint8_t)T_SOLID;
        if (row_in) {
            m_next = (WALLS && p.any_solid_link) ? p.mask[n] : 0u;
            fl_next = p.flags[n];
        }
        cp_async_wait<1>();
        __syncthreads();
        for (int z = z0; z < z1; ++z, n += area) {
            const uint32_t m = m_next;
            const uint8_t fl = fl_next;
            if (row_in && z + 1 < z1) {
                m_next = (WALLS && p.any_solid_link) ? p.mask[n + area] : 0u;
                fl_next = p.flags[n + area];
            }
            float* pm = ring + tile_slot(z - 1) * kTilePlaneFloats;
            float* p0 = ring + tile_slot(z) * kTilePlaneFloats;
            float* pp = ring + tile_slot(z + 1) * kTilePlaneFloats;
            uint32_t* bm = bits + tile_slot(z - 1) * kTileRecords;
            uint32_t* b0 = bits + tile_slot(z) * kTileRecords;
            uint32_t* bp = bits + tile_slot(z + 1) * kTileRecords;
            if (row_in) {
                if ((fl & (TYPE_MASK | F_SPECIAL)) == T_FLUID) {
                    float h[19];
                    tile_odd_gather(pm, p0, pp, own, m, h);
                    collide<BODY>(h, p);
                    tile_odd_scatter<FORCE, WALLS>(pm, p0, pp, bm, b0, bp, own, rid, m, h, fx, fy, fz);
                } else if (p.any_inlet && (fl & TYPE_MASK) == T_INLET) {
                    tile_odd_produce<WALLS>(p, pm, p0, pp, bm, b0, bp, own, rid, x, y, z);
                }
            }
            __syncthreads();  // plane z is scattered: plane z - 1 is final
            if (WALLS)
                tile_odd_writeback(p, A, pm, bm, x0, y0, z - 1, z - 1 > z0 && z - 1 < z1 - 1);
            else
                tile_odd_writeback_static(p, A, pm, x0, y0, z - 1,
                                          tile_axis_mask<2>(z - 1 - z0, z1 - z0),
                                          z - 1 > z0 && z - 1 < z1 - 1, owned);
            __syncthreads();  // the slot of z - 1 is free again
            if (z + 3 <= z1)
                tile_load_plane(p, A, ring + tile_slot(z + 3) * kTilePlaneFloats, x0, y0,
                                tile_wrap(z + 3, p.nz), false);
            cp_async_commit();
            cp_async_wait<1>();  // plane z + 2 has arrived (z + 3 may still be in flight)
            __syncthreads();
        }
        // the chunk's last plane and the halo plane after it
        for (int pl = z1 - 1; pl <= z1; ++pl) {
            const float* ring_s = ring + tile_slot(pl) * kTilePlaneFloats;
            if (WALLS)
                tile_odd_writeback(p, A, ring_s, bits + tile_slot(pl) * kTileRecords, x0, y0, pl, false);
            else
                tile_odd_writeback_static(p, A, ring_s, x0, y0, pl,
                                          tile_axis_mask<2>(pl - z0, z1 - z0), false, owned);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

}  // namespace lbm
