// Kernels of the D3Q19 BGK step, templated on the population layout L.  Included by one
// translation unit per layout, which instantiates them and defines the launch functions.
//
// Cell kernels use a 3D grid: threads along x (blockDim.x), rows along y (blockDim.y), one z
// plane per blockIdx.z; a thread owns cell n = x + nx (y + ny z).
//
// The per-link rules, the same in every scheme ("GPU lattice Boltzmann: streaming layout and
// performance", paragraph after the layout bullets): population q of FLUID cell x comes from
// s = x - c_q (wrapped on periodic axes, clamped onto the last layer beyond an OPEN face):
// FLUID s streams its post-collision value, SOLID s reflects x's own post-collision population
// opposite(q) (halfway bounce-back, PortLBM §3.1), INLET s supplies f_eq(rho_in, u_in), a
// MOVING_WALL s reflects like SOLID plus 2 w_q (c_q.u_w) / c_s^2 (the mirror method of
// "GPU加速LBM流体仿真" §4.2, at the reference density 1).
#pragma once

#include <type_traits>

#include "lbm_device.cuh"

namespace lbm {

struct Link {
    uint32_t cell;
    int face;  // -1: inside the domain; otherwise 2*axis + side of the first axis clamped
};

// Cell x + d with the face rules; `face` records the first axis (x, then y, then z) whose
// coordinate lay beyond an OPEN face.
__device__ __forceinline__ Link link_cell(const Params& p, int x, int y, int z, int dx, int dy,
                                          int dz) {
    int face = -1;
    int v = x + dx;
    if (v < 0) { if (p.open[0]) { v = 0; face = 0; } else v += p.nx; }
    else if (v >= p.nx) { if (p.open[0]) { v = p.nx - 1; face = 1; } else v -= p.nx; }
    int w = y + dy;
    if (w < 0) { if (p.open[1]) { w = 0; if (face < 0) face = 2; } else w += p.ny; }
    else if (w >= p.ny) { if (p.open[1]) { w = p.ny - 1; if (face < 0) face = 3; } else w -= p.ny; }
    int u = z + dz;
    if (u < 0) { if (p.open[2]) { u = 0; if (face < 0) face = 4; } else u += p.nz; }
    else if (u >= p.nz) { if (p.open[2]) { u = p.nz - 1; if (face < 0) face = 5; } else u -= p.nz; }
    Link l;
    l.cell = (uint32_t)v + (uint32_t)p.nx * ((uint32_t)w + (uint32_t)p.ny * (uint32_t)u);
    l.face = face;
    return l;
}

// Position of cell (x, y, z) on the face layers of `axis` (row-major over the other two axes).
__device__ __forceinline__ size_t face_pos(const Params& p, int axis, int x, int y, int z) {
    return axis == 0 ? (size_t)y + (size_t)p.ny * z
         : axis == 1 ? (size_t)x + (size_t)p.nx * z : (size_t)x + (size_t)p.nx * y;
}
__device__ __forceinline__ size_t face_area(const Params& p, int axis) {
    return axis == 0 ? (size_t)p.ny * p.nz : axis == 1 ? (size_t)p.nx * p.nz : (size_t)p.nx * p.ny;
}
__device__ __forceinline__ size_t scratch_slot(const Params& p, int face, int q, int x, int y,
                                               int z) {
    const int axis = face >> 1;
    return p.face_base[axis][face & 1] + (size_t)q * face_area(p, axis) + face_pos(p, axis, x, y, z);
}

// Neighbour cell indices n + d, with d the sum of one per-axis delta per velocity component:
// wrapped on PERIODIC axes; with `clamp` (the A-B pulls) clamped onto the last layer on OPEN axes,
// the zero-gradient source of a pull.  The AA odd kernels wrap everywhere: a cell whose link
// crosses an OPEN face is special there and takes no such link in the main kernel.  `clamp` is a
// constant at every call site.
__device__ __forceinline__ int edge_delta(int at, int n, int stride, bool open, int c) {
    if (c < 0) return at == 0 ? (open ? 0 : (n - 1) * stride) : -stride;
    return at == n - 1 ? (open ? 0 : -(n - 1) * stride) : stride;
}
struct Nbr {
    int dx[3], dy[3], dz[3];  // delta for c = -1, 0, +1 along each axis
    __device__ __forceinline__ Nbr(const Params& p, int x, int y, int z, bool clamp) {
        const int sx = 1, sy = p.nx, sz = p.nx * p.ny;
        dx[0] = edge_delta(x, p.nx, sx, clamp && p.open[0], -1);
        dx[1] = 0;
        dx[2] = edge_delta(x, p.nx, sx, clamp && p.open[0], 1);
        dy[0] = edge_delta(y, p.ny, sy, clamp && p.open[1], -1);
        dy[1] = 0;
        dy[2] = edge_delta(y, p.ny, sy, clamp && p.open[1], 1);
        dz[0] = edge_delta(z, p.nz, sz, clamp && p.open[2], -1);
        dz[1] = 0;
        dz[2] = edge_delta(z, p.nz, sz, clamp && p.open[2], 1);
    }
    // cell n + s c_q, s = +1 or -1
    template <int Q, int S>
    __device__ __forceinline__ uint32_t at(uint32_t n) const {
        return n + (uint32_t)(dx[S * cx(Q) + 1] + dy[S * cy(Q) + 1] + dz[S * cz(Q) + 1]);
    }
};

// Momentum exchange of a FLUID cell: every link along which post-collision population q bounces
// back (bit q of the solid-link mask: x + c_q, wrapped or clamped, is SOLID) adds 2 c_q f*_q,
// f* = h* + w.
template <int Q>
__device__ __forceinline__ void accumulate_force(float h_post, float& fx, float& fy, float& fz) {
    const float t = 2.0f * (h_post + wq(Q));
    if (cx(Q) > 0) fx += t; else if (cx(Q) < 0) fx -= t;
    if (cy(Q) > 0) fy += t; else if (cy(Q) < 0) fy -= t;
    if (cz(Q) > 0) fz += t; else if (cz(Q) < 0) fz -= t;
}

// Post-collision population Q of one cell: from a one-cell array, or from lane LANE (0: the even
// cell, 1: the odd cell) of a two-cell array.
template <int Q>
__device__ __forceinline__ float pop(const float (&h)[19]) { return h[Q]; }
template <int LANE>
struct PairLane {
    const float2 (&h)[19];
};
template <int Q, int LANE>
__device__ __forceinline__ float pop(const PairLane<LANE>& l) { return LANE ? l.h[Q].y : l.h[Q].x; }

template <int Q = 1, typename H>
__device__ __forceinline__ void mask_forces(uint32_t m, const H& h, float& fx, float& fy, float& fz) {
    if ((m >> Q) & 1u) accumulate_force<Q>(pop<Q>(h), fx, fy, fz);
    if constexpr (Q < 18) mask_forces<Q + 1>(m, h, fx, fy, fz);
}

// Momentum exchange of the MOVING_WALL links of a special cell: what the fluid gives up on link q
// is c_q (f*_q + f_back), f_back = f*_q + 6 w (c_opp(q).u_w), i.e. c_q (2 f*_q - 6 w_q (c_q.u_w)).
template <int Q = 1, typename H>
__device__ __forceinline__ void moving_forces(const Params& p, const H& h, int x, int y, int z,
                                              float& fx, float& fy, float& fz) {
    const Link d = link_cell(p, x, y, z, cx(Q), cy(Q), cz(Q));
    if ((p.flags[d.cell] & TYPE_MASK) == T_MOVING) {
        const float t = 2.0f * (pop<Q>(h) + wq(Q)) - p.wterm[Q];
        if (cx(Q) > 0) fx += t; else if (cx(Q) < 0) fx -= t;
        if (cy(Q) > 0) fy += t; else if (cy(Q) < 0) fy -= t;
        if (cz(Q) > 0) fz += t; else if (cz(Q) < 0) fz -= t;
    }
    if constexpr (Q < 18) moving_forces<Q + 1>(p, h, x, y, z, fx, fy, fz);
}

template <int Q>
__device__ __forceinline__ bool solid_link(uint32_t m) { return (m >> Q) & 1u; }

// Thread -> cell of the 3D launch; false for the ragged tail.
struct CellCoord {
    int x, y, z;
    uint32_t n;
};
// PLANES: the plane from zbase / zstep (the A-B step kernels, which also run over some planes)
template <bool PLANES = false>
__device__ __forceinline__ bool grid_cell(const Params& p, CellCoord& c) {
    c.x = blockIdx.x * blockDim.x + threadIdx.x;
    c.y = blockIdx.y * blockDim.y + threadIdx.y;
    if constexpr (PLANES) c.z = p.zbase + p.zstep * (int)blockIdx.z;
    else c.z = p.zrev ? p.nz - 1 - (int)blockIdx.z : (int)blockIdx.z;
    c.n = (uint32_t)c.x + (uint32_t)p.nx * ((uint32_t)c.y + (uint32_t)p.ny * c.z);
    return c.x < p.nx && c.y < p.ny;
}
// Thread -> i-th special cell of the 1D boundary launch.
__device__ __forceinline__ bool special_cell(const Params& p, CellCoord& c) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n_special) return false;
    c.n = p.special[i];
    c.x = (int)(c.n % (uint32_t)p.nx);
    c.y = (int)((c.n / (uint32_t)p.nx) % (uint32_t)p.ny);
    c.z = (int)(c.n / ((uint32_t)p.nx * (uint32_t)p.ny));
    return true;
}

// ============================== AA pattern, even step ===========================================
// "In place" bullet: read population q of x at (q, x); write the collided one at (opposite(q), x).
// Purely local, so every FLUID cell (special ones included) is handled here.
// Hot-path addressing: element offset of cell n relative to a population's plane pointer
// (I = uint32_t when every element offset of the buffer fits in 32 bits, else long long).
template <int L, typename I>
__device__ __forceinline__ I cell_off(int q, uint32_t n) {
    return (I)n * (I)cell_stride<L>(q);
}

template <int L, bool FORCE, bool BODY, typename I>
__global__ void __launch_bounds__(256) k_aa_even(Params p) {
    CellCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (grid_cell(p, c)) {
        const uint8_t fl = p.flags[c.n];
        if ((fl & TYPE_MASK) == T_FLUID) {
            float h[19];
#pragma unroll
            for (int q = 0; q < 19; ++q) h[q] = ld<L>(p.pa[q], cell_off<L, I>(q, c.n));
            collide<BODY>(h, p);
            // store addresses formed after the collision, not kept from the loads
            uint32_t ns = c.n;
            asm volatile("" : "+r"(ns) : "f"(h[0]), "f"(h[18]));
#pragma unroll
            for (int q = 0; q < 19; ++q) st<L>(p.pa[opp(q)], cell_off<L, I>(q, ns), h[q]);
            if (FORCE && !(fl & F_BULK)) {
                mask_forces(p.mask[c.n], h, fx, fy, fz);
                if (p.any_moving && (fl & F_SPECIAL)) moving_forces(p, h, c.x, c.y, c.z, fx, fy, fz);
            }
        } else if (p.any_inlet && (fl & TYPE_MASK) == T_INLET) {
            // an INLET cell's post-collision state is the reservoir's f_eq(rho_in, u_in)
#pragma unroll
            for (int q = 0; q < 19; ++q) st<L>(p.pa[opp(q)], cell_off<L, I>(q, c.n), p.heq_in[q]);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// The steps in which a cell reads and writes only its own populations -- the AA even step, and the
// A-B collision of the natural state -- in the collision layout, with each warp's cells staged
// through shared memory.  The 19-population records of a warp's consecutive cells are one
// contiguous run ([PortLBM] §3.2, Fig. 2), so the warp copies it in and out in coalesced runs and
// each lane then reads and writes its own record in shared memory (a stride of 19 words, odd: no
// bank conflicts); element loads strided by the 76-byte record touched 19 times as many sectors
// per request (even step 0.173 -> 0.056 ms at 128^3).  The bundle layout's stride-3 element
// accesses measured faster unstaged.  OPP: the AA even step (the collided population q goes to
// opposite(q)); else the A-B collision (to q, in B, which may equal A).  An INLET cell stores the
// reservoir's f_eq(rho_in, u_in); any other cell that is not FLUID keeps what was loaded.
template <bool FORCE, bool BODY, bool OPP>
__global__ void __launch_bounds__(256) k_own_staged(Params p) {
    constexpr int L = LAYOUT_COLLISION;
    __shared__ float tile[kWarpsPerBlock][32 * 19];
    CellCoord c;
    const bool in = grid_cell<true>(p, c);
    const int lane = threadIdx.x & 31;
    const int warp = (threadIdx.x + blockDim.x * threadIdx.y) >> 5;
    // the warp's cells: lanes [0, cnt) of one row (blockDim.x is a multiple of 32), consecutive
    // cell indices from n0, whose records are elements [19 n0, 19 (n0 + cnt))
    const int cnt = __popc(__ballot_sync(0xffffffffu, in));
    const uint32_t n0 = __shfl_sync(0xffffffffu, c.n, 0);
    float* t = tile[warp];
    const float* src = static_cast<const float*>(p.A) + (size_t)n0 * 19;
    float* dst = static_cast<float*>(OPP ? p.A : p.B) + (size_t)n0 * 19;
    for (int k = lane; k < cnt * 19; k += 32) t[k] = src[k];
    __syncwarp();
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const uint8_t fl = in ? p.flags[c.n] : (uint8_t)T_SOLID;
    if ((fl & TYPE_MASK) == T_FLUID) {
        float h[19];
#pragma unroll
        for (int q = 0; q < 19; ++q) h[q] = t[idx<L, int>(q, (uint32_t)lane, 32)];
        collide<BODY>(h, p);
#pragma unroll
        for (int q = 0; q < 19; ++q) t[idx<L, int>(OPP ? opp(q) : q, (uint32_t)lane, 32)] = h[q];
        if (FORCE && !(fl & F_BULK)) {
            mask_forces(p.mask[c.n], h, fx, fy, fz);
            if (p.any_moving && (fl & F_SPECIAL)) moving_forces(p, h, c.x, c.y, c.z, fx, fy, fz);
        }
    } else if (p.any_inlet && (fl & TYPE_MASK) == T_INLET) {
        // INLET producer: the reservoir's f_eq(rho_in, u_in) as its post-collision state
#pragma unroll
        for (int q = 0; q < 19; ++q) t[idx<L, int>(OPP ? opp(q) : q, (uint32_t)lane, 32)] = p.heq_in[q];
    }
    __syncwarp();
    for (int k = lane; k < cnt * 19; k += 32) dst[k] = t[k];
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

// ============================== AA pattern, odd step ============================================
// "In place" bullet: read population q of x at (opposite(q), x - c_q); write the collided value at
// (q, x + c_q).  Cell x reads and writes exactly the same 19 slots, so cells never race.  A link
// whose partner cell is SOLID uses x's own mirrored slot instead: the gather of q reads (q, x),
// which holds f*_opposite(q)(x) after the even step, and the scatter of q writes (opposite(q), x).
//
// Main kernel: FLUID cells that are not special.  The solid-link mask selects, per population,
// between the neighbour's slot and the cell's own mirrored slot, so bulk and near-wall cells run
// the same branch-free code.
// I = uint32_t: one base and 32-bit element offsets (fewer instructions per access); otherwise
// per-population plane pointers with 64-bit offsets.
template <int L, typename I, int Q = 0>
__device__ __forceinline__ void aa_odd_load(const Params& p, const Nbr& nb, uint32_t n, uint32_t m,
                                            float (&h)[19]) {
    constexpr uint32_t S = cell_stride<L>(Q);
    if constexpr (std::is_same<I, uint32_t>::value) {
        // own slot (q, x); neighbour slot (opp q, x - c_q)
        const uint32_t own = p.plane32[Q] + n * S;
        const uint32_t far = p.plane32[opp(Q)] + nb.template at<Q, -1>(n) * S;
        h[Q] = ld<L>(p.A, solid_link<opp(Q)>(m) ? own : far);
    } else {
        const I own = (I)p.pdiff[Q] + cell_off<L, I>(Q, n);
        const I far = cell_off<L, I>(Q, nb.template at<Q, -1>(n));
        h[Q] = ld<L>(p.pa[opp(Q)], solid_link<opp(Q)>(m) ? own : far);
    }
    if constexpr (Q < 18) aa_odd_load<L, I, Q + 1>(p, nb, n, m, h);
}

template <int L, typename I, bool FORCE, int Q = 0>
__device__ __forceinline__ void aa_odd_store(const Params& p, const Nbr& nb, uint32_t n, uint32_t m,
                                             const float (&h)[19], float& fx, float& fy,
                                             float& fz) {
    // own slot (opp q, x); neighbour slot (q, x + c_q); a bounced link also carries its
    // momentum-exchange term
    constexpr uint32_t S = cell_stride<L>(Q);
    const bool bounce = solid_link<Q>(m);
    if constexpr (std::is_same<I, uint32_t>::value) {
        const uint32_t own = p.plane32[opp(Q)] + n * S;
        const uint32_t far = p.plane32[Q] + nb.template at<Q, 1>(n) * S;
        st<L>(p.A, bounce ? own : far, h[Q]);
    } else {
        const I own = cell_off<L, I>(Q, n) - (I)p.pdiff[Q];
        const I far = cell_off<L, I>(Q, nb.template at<Q, 1>(n));
        st<L>(p.pa[Q], bounce ? own : far, h[Q]);
    }
    if (FORCE && Q > 0 && bounce) accumulate_force<Q>(h[Q], fx, fy, fz);
    if constexpr (Q < 18) aa_odd_store<L, I, FORCE, Q + 1>(p, nb, n, m, h, fx, fy, fz);
}

// INLET cells are producers in the AA odd step ("PortLBM", §3.1, last paragraph: the inlet imposes
// the equilibrium): population q of the reservoir, f_eq,q(rho_in, u_in), goes to (q, s + c_q), the
// slot in which a FLUID cell's scatter leaves its population q for the neighbour's next even step.
// A link that leaves the domain through an OPEN face reaches nobody and is dropped (its wrapped
// slot belongs to the zero-gradient copies of the boundary kernel).  The rest population stays.
__device__ __forceinline__ bool leaves_open(const Params& p, int x, int y, int z, int c_x, int c_y,
                                            int c_z) {
    return (p.open[0] && ((c_x < 0 && x == 0) || (c_x > 0 && x == p.nx - 1))) ||
           (p.open[1] && ((c_y < 0 && y == 0) || (c_y > 0 && y == p.ny - 1))) ||
           (p.open[2] && ((c_z < 0 && z == 0) || (c_z > 0 && z == p.nz - 1)));
}
template <int L, typename I, int Q = 1>
__device__ __forceinline__ void aa_odd_produce(const Params& p, const Nbr& nb, uint32_t n, int x,
                                               int y, int z) {
    constexpr uint32_t S = cell_stride<L>(Q);
    if (!leaves_open(p, x, y, z, cx(Q), cy(Q), cz(Q))) {
        if constexpr (std::is_same<I, uint32_t>::value)
            st<L>(p.A, p.plane32[Q] + nb.template at<Q, 1>(n) * S, p.heq_in[Q]);
        else
            st<L>(p.pa[Q], cell_off<L, I>(Q, nb.template at<Q, 1>(n)), p.heq_in[Q]);
    }
    if constexpr (Q < 18) aa_odd_produce<L, I, Q + 1>(p, nb, n, x, y, z);
}

template <int L, bool FORCE, bool BODY, typename I>
__global__ void __launch_bounds__(256) k_aa_odd(Params p) {
    CellCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (grid_cell(p, c)) {
        // the mask is loaded beside the flag byte, not after it (one round trip less)
        const uint32_t m = p.any_solid_link ? p.mask[c.n] : 0u;
        const uint8_t fl = p.flags[c.n];
        if ((fl & (TYPE_MASK | F_SPECIAL)) == T_FLUID) {
            const Nbr nb(p, c.x, c.y, c.z, false);
            float h[19];
            aa_odd_load<L, I>(p, nb, c.n, m, h);
            collide<BODY>(h, p);
            // the store addresses are formed after the collision (keeps them out of registers
            // while the loads are in flight)
            uint32_t ns = c.n, ms = m;
            asm volatile("" : "+r"(ns), "+r"(ms) : "f"(h[0]), "f"(h[18]));
            aa_odd_store<L, I, FORCE>(p, nb, ns, ms, h, fx, fy, fz);
        } else if (p.any_inlet && (fl & TYPE_MASK) == T_INLET) {
            const Nbr nb(p, c.x, c.y, c.z, false);
            aa_odd_produce<L, I>(p, nb, c.n, c.x, c.y, c.z);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// The boundary kernels of the AA odd and A-B pull steps (special cells, general per-link rules)
// are in lbm_kernels_boundary.cuh.

// Open-face pre-gather for the AA odd step: for every FLUID cell x on face layer (axis, side) and
// every q whose source x - c_q lies beyond that face first, copy the clamped source's
// post-collision population q -- at (opposite(q), s) -- into scratch, before the odd kernels
// overwrite that slot.  Only the 5 velocities with c_axis pointing into the domain from that face
// (+1 on the low side, -1 on the high side) can have such a source: one thread per (k, face cell),
// k-th of those velocities.
__device__ __forceinline__ int face_velocity(int axis, int sgn, int k) {
    int cnt = 0;
    for (int q = 1; q < 19; ++q) {
        const int c = axis == 0 ? cx_rt(q) : axis == 1 ? cy_rt(q) : cz_rt(q);
        if (c == sgn) {
            if (cnt == k) return q;
            ++cnt;
        }
    }
    return 0;
}

// One launch for every open face: blockIdx.y = 2 * axis + side.
template <int L>
__global__ void __launch_bounds__(256) k_pregather(Params p) {
    const int axis = (int)blockIdx.y >> 1, side = (int)blockIdx.y & 1;
    if (!p.open[axis]) return;
    const size_t area = face_area(p, axis);
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 5 * area) return;
    const int k = (int)(i / area);
    const size_t pos = i - (size_t)k * area;
    const int q = face_velocity(axis, side ? -1 : 1, k);
    int x, y, z;
    if (axis == 0) { x = side ? p.nx - 1 : 0; y = (int)(pos % p.ny); z = (int)(pos / p.ny); }
    else if (axis == 1) { y = side ? p.ny - 1 : 0; x = (int)(pos % p.nx); z = (int)(pos / p.nx); }
    else { z = side ? p.nz - 1 : 0; x = (int)(pos % p.nx); y = (int)(pos / p.nx); }
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    if ((p.flags[n] & TYPE_MASK) != T_FLUID) return;
    const Link s = link_cell(p, x, y, z, -cx_rt(q), -cy_rt(q), -cz_rt(q));
    if (s.face != 2 * axis + side) return;
    if ((p.flags[s.cell] & TYPE_MASK) != T_FLUID) return;
    p.scratch[p.face_base[axis][side] + (size_t)q * area + pos] = ld<L>(p.A, idx_rt<L>(opp(q), s.cell, p.N));
}

// ============================== two buffers (A-B) ===============================================
// Pull (PortLBM §3.3 one-step pull, two lattices): gather the 19 incoming populations from the
// neighbours' post-collision values in A -- SOLID source: x's own opposite population, at
// (opposite(q), x) -- collide, and write the post-collision values to B at (q, x).
template <int L, typename I, int Q = 0>
__device__ __forceinline__ void ab_load(const Params& p, const Nbr& nb, uint32_t n, uint32_t m,
                                        float (&h)[19]) {
    // own slot (opp q, x); neighbour slot (q, x - c_q)
    constexpr uint32_t S = cell_stride<L>(Q);
    if constexpr (std::is_same<I, uint32_t>::value) {
        const uint32_t own = p.plane32[opp(Q)] + n * S;
        const uint32_t far = p.plane32[Q] + nb.template at<Q, -1>(n) * S;
        h[Q] = ld<L>(p.A, solid_link<opp(Q)>(m) ? own : far);
    } else {
        const I own = cell_off<L, I>(Q, n) - (I)p.pdiff[Q];
        const I far = cell_off<L, I>(Q, nb.template at<Q, -1>(n));
        h[Q] = ld<L>(p.pa[Q], solid_link<opp(Q)>(m) ? own : far);
    }
    if constexpr (Q < 18) ab_load<L, I, Q + 1>(p, nb, n, m, h);
}

// general per-link gather (special cells)
template <int L, int Q = 0>
__device__ __forceinline__ void ab_gather_all(const Params& p, float (&h)[19], uint32_t n, int x,
                                              int y, int z) {
    const Link s = link_cell(p, x, y, z, -cx(Q), -cy(Q), -cz(Q));
    const int t = p.flags[s.cell] & TYPE_MASK;
    if (t == T_SOLID) h[Q] = ld<L>(p.A, idx<L>(opp(Q), n, p.N));
    else if (t == T_MOVING) h[Q] = ld<L>(p.A, idx<L>(opp(Q), n, p.N)) + p.wterm[Q];
    else if (t == T_INLET) h[Q] = p.heq_in[Q];
    else h[Q] = ld<L>(p.A, idx<L>(Q, s.cell, p.N));
    if constexpr (Q < 18) ab_gather_all<L, Q + 1>(p, h, n, x, y, z);
}

// FROM_NATURAL: collide the natural state of the cell (first step after a state load, and the
// first pass of the two-pass scheme, where B may equal A); every FLUID cell.  Otherwise
// pull-collide for the FLUID cells that are not special.
// 6 resident blocks per SM (<= 40 registers, no spills): measured faster for the pull
template <int L, bool FORCE, bool BODY, bool FROM_NATURAL, typename I>
__global__ void __launch_bounds__(256, 6) k_ab(Params p) {
    CellCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (grid_cell<true>(p, c)) {
        // the natural-state collision needs the links only for the force; the mask is loaded
        // beside the flag byte, not after it
        const uint32_t m = (p.any_solid_link && (FORCE || !FROM_NATURAL)) ? p.mask[c.n] : 0u;
        const uint8_t fl = p.flags[c.n];
        const uint8_t want = FROM_NATURAL ? TYPE_MASK : (TYPE_MASK | F_SPECIAL);
        if ((fl & want) == T_FLUID) {
            float h[19];
            if (FROM_NATURAL) {
#pragma unroll
                for (int q = 0; q < 19; ++q) h[q] = ld<L>(p.pa[q], cell_off<L, I>(q, c.n));
            } else {
                const Nbr nb(p, c.x, c.y, c.z, true);
                ab_load<L, I>(p, nb, c.n, m, h);
            }
            collide<BODY>(h, p);
            uint32_t ns = c.n;
            asm volatile("" : "+r"(ns) : "f"(h[0]), "f"(h[18]));
#pragma unroll
            for (int q = 0; q < 19; ++q) st<L>(p.pb[q], cell_off<L, I>(q, ns), h[q]);
            if (FORCE && m) mask_forces(m, h, fx, fy, fz);
            if (FORCE && FROM_NATURAL && p.any_moving && (fl & F_SPECIAL))
                moving_forces(p, h, c.x, c.y, c.z, fx, fy, fz);
        } else if (p.any_inlet && (fl & TYPE_MASK) == T_INLET) {
            // INLET producer: its post-collision state, where the pulls read it, is f_eq(rho_in,
            // u_in) (written in place too: the two-pass scheme's streaming reads it there)
#pragma unroll
            for (int q = 0; q < 19; ++q) st<L>(p.pb[q], cell_off<L, I>(q, c.n), p.heq_in[q]);
        } else if ((fl & TYPE_MASK) != T_FLUID && p.pb[0] != p.pa[0]) {
            // SOLID and MOVING_WALL slots are never read; writing them keeps every 32-byte sector
            // of the destination fully written (no fill from DRAM for partly written sectors)
#pragma unroll
            for (int q = 0; q < 19; ++q) st<L>(p.pb[q], cell_off<L, I>(q, c.n), 0.0f);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

// A-B pull in the collision and bundle layouts, with the stores staged: each lane gathers and
// collides its cell as `k_ab` does (element loads from the neighbours' records), writes its
// populations into the warp's shared-memory tile (the layout for N = 32), and the warp writes its
// cells' records to B in coalesced runs -- one run (collision) or one per bundle -- instead of
// element stores 76 or 12 bytes apart.  INLET cells get the reservoir's f_eq(rho_in, u_in); the
// other cells that are not pulled here (SOLID, MOVING_WALL, special) get zeros, so every sector of
// B is written whole; the boundary kernel, launched after this one, overwrites the special cells'
// records.
template <int L, bool FORCE, bool BODY, typename I>
__global__ void __launch_bounds__(256) k_ab_pull_staged(Params p) {
    __shared__ float tile[kWarpsPerBlock][32 * 19];
    CellCoord c;
    const bool in = grid_cell<true>(p, c);
    const int lane = threadIdx.x & 31;
    const int warp = (threadIdx.x + blockDim.x * threadIdx.y) >> 5;
    const int cnt = __popc(__ballot_sync(0xffffffffu, in));
    const uint32_t n0 = __shfl_sync(0xffffffffu, c.n, 0);
    float* t = tile[warp];
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const uint32_t m = (in && p.any_solid_link) ? p.mask[c.n] : 0u;
    const uint8_t fl = in ? p.flags[c.n] : (uint8_t)T_SOLID;
    if ((fl & (TYPE_MASK | F_SPECIAL)) == T_FLUID) {
        const Nbr nb(p, c.x, c.y, c.z, true);
        float h[19];
        ab_load<L, I>(p, nb, c.n, m, h);
        collide<BODY>(h, p);
#pragma unroll
        for (int q = 0; q < 19; ++q) t[idx<L, int>(q, (uint32_t)lane, 32)] = h[q];
        if (FORCE && m) mask_forces(m, h, fx, fy, fz);
    } else {
        // INLET producer: f_eq(rho_in, u_in); zeros for the others
        const bool inl = p.any_inlet && (fl & TYPE_MASK) == T_INLET;
#pragma unroll
        for (int q = 0; q < 19; ++q) t[idx<L, int>(q, (uint32_t)lane, 32)] = inl ? p.heq_in[q] : 0.0f;
    }
    __syncwarp();
    float* B = static_cast<float*>(p.B);
#pragma unroll
    for (int q = 0; q < 19; ++q) {
        // one run per record group: the collision layout's records, or a bundle (from its first
        // member q: bundle offset in units of N, members per cell)
        if ((L == LAYOUT_COLLISION && q == 0) || (L != LAYOUT_COLLISION && bundle_j(q) == 0)) {
            const int off = L == LAYOUT_COLLISION ? 0 : bundle_off(q);
            const int m = L == LAYOUT_COLLISION ? 19 : bundle_size(q);
            float* dst = B + (size_t)off * p.N + (size_t)n0 * m;
            for (int k = lane; k < cnt * m; k += 32) dst[k] = t[32 * off + k];
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

// Streaming only: natural state into B from the post-collision state in A (second pass of the
// two-pass scheme).  Main kernel (non-special FLUID cells) and boundary kernel (special cells).
template <int L, typename I>
__global__ void __launch_bounds__(256) k_stream(Params p) {
    CellCoord c;
    if (!grid_cell(p, c)) return;
    const uint32_t m = p.any_solid_link ? p.mask[c.n] : 0u;
    const uint8_t fl = p.flags[c.n];
    if ((fl & TYPE_MASK) != T_FLUID) {
        // SOLID / MOVING_WALL slots are never read; INLET slots are refilled by the next step's
        // collision pass before any pull reads them: zeros keep the destination's sectors whole
#pragma unroll
        for (int q = 0; q < 19; ++q) st<L>(p.pb[q], cell_off<L, I>(q, c.n), 0.0f);
        return;
    }
    if (fl & F_SPECIAL) return;
    const Nbr nb(p, c.x, c.y, c.z, true);
    float h[19];
    ab_load<L, I>(p, nb, c.n, m, h);
#pragma unroll
    for (int q = 0; q < 19; ++q) st<L>(p.pb[q], cell_off<L, I>(q, c.n), h[q]);
}

template <int L>
__global__ void __launch_bounds__(256) k_stream_special(Params p) {
    CellCoord c;
    if (!special_cell(p, c)) return;
    float h[19];
    ab_gather_all<L>(p, h, c.n, c.x, c.y, c.z);
#pragma unroll
    for (int q = 0; q < 19; ++q) st<L>(p.B, idx<L>(q, c.n, p.N), h[q]);
}

// ============================== state access off the step path ==================================
// Natural shifted population q of FLUID cell (x, y, z) for a buffer in state `state`.
template <int L>
__device__ __forceinline__ float natural_h(const Params& p, int state, int q, uint32_t n, int x,
                                           int y, int z) {
    if (state == ST_NATURAL) return ld<L>(p.A, idx_rt<L>(q, n, p.N));
    const Link s = link_cell(p, x, y, z, -cx(q), -cy(q), -cz(q));
    const int t = p.flags[s.cell] & TYPE_MASK;
    if (t == T_INLET) return p.heq_in[q];
    const float wall = t == T_MOVING ? p.wterm[q] : 0.0f;
    if (state == ST_POST_AA) {
        if (t == T_SOLID || t == T_MOVING) return ld<L>(p.A, idx_rt<L>(q, n, p.N)) + wall;
        return ld<L>(p.A, idx_rt<L>(opp(q), s.cell, p.N));
    }
    if (t == T_SOLID || t == T_MOVING) return ld<L>(p.A, idx_rt<L>(opp(q), n, p.N)) + wall;
    return ld<L>(p.A, idx_rt<L>(q, s.cell, p.N));
}

// Canonical absolute f[q*N + n] for flat indices [i0, i0 + count) into out[0, count).
template <int L>
__global__ void __launch_bounds__(256) k_unpack(Params p, int state, float* out, size_t i0,
                                                size_t count) {
    const size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= count) return;
    const size_t i = i0 + k;
    const int q = (int)(i / p.N);
    const uint32_t n = (uint32_t)(i - (size_t)q * p.N);
    const int x = (int)(n % (uint32_t)p.nx);
    const int y = (int)((n / (uint32_t)p.nx) % (uint32_t)p.ny);
    const int z = (int)(n / ((uint32_t)p.nx * (uint32_t)p.ny));
    const int t = p.flags[n] & TYPE_MASK;
    float v;
    if (t == T_SOLID || t == T_MOVING) v = 0.0f;
    else if (t == T_INLET) v = p.heq_in[q] + wq(q);
    else v = natural_h<L>(p, state, q, n, x, y, z) + wq(q);
    out[k] = v;
}

// Canonical absolute f[q*N + n], flat indices [i0, i0 + count), into the natural shifted state.
template <int L>
__global__ void __launch_bounds__(256) k_pack(Params p, const float* in, size_t i0, size_t count) {
    const size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= count) return;
    const size_t i = i0 + k;
    const int q = (int)(i / p.N);
    const uint32_t n = (uint32_t)(i - (size_t)q * p.N);
    st<L>(p.A, idx_rt<L>(q, n, p.N), in[k] - wq(q));
}

// Natural shifted state f_eq(rho, u) - w for cells [n0, n0 + count).
template <int L>
__global__ void __launch_bounds__(256) k_equilibrium(Params p, const float* rho, const float* u0,
                                                     const float* u1, const float* u2,
                                                     uint32_t n0, uint32_t count) {
    const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= count) return;
    const uint32_t n = n0 + k;
    const float r = rho[k], ux = u0[k], uy = u1[k], uz = u2[k];
    const float drho = r - 1.0f;
    const float uu15 = 1.5f * (ux * ux + uy * uy + uz * uz);
#pragma unroll
    for (int q = 0; q < 19; ++q) {
        const float cu = (float)cx(q) * ux + (float)cy(q) * uy + (float)cz(q) * uz;
        const float poly = fmaf(cu, fmaf(4.5f, cu, 3.0f), -uu15);
        st<L>(p.A, idx<L>(q, n, p.N), wq(q) * fmaf(r, poly, drho));
    }
}

// rho and u (Guo-shifted) of the natural state for cells [n0, n0 + count).
template <int L>
__global__ void __launch_bounds__(256) k_macro(Params p, int state, float rho_in, float ux_in,
                                               float uy_in, float uz_in, float* rho, float* u0,
                                               float* u1, float* u2, uint32_t n0, uint32_t count) {
    const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= count) return;
    const uint32_t n = n0 + k;
    const int t = p.flags[n] & TYPE_MASK;
    if (t == T_SOLID) { rho[k] = 0.f; u0[k] = u1[k] = u2[k] = 0.f; return; }
    if (t == T_MOVING) { rho[k] = 1.f; u0[k] = p.uw[0]; u1[k] = p.uw[1]; u2[k] = p.uw[2]; return; }
    if (t == T_INLET) { rho[k] = rho_in; u0[k] = ux_in; u1[k] = uy_in; u2[k] = uz_in; return; }
    const int x = (int)(n % (uint32_t)p.nx);
    const int y = (int)((n / (uint32_t)p.nx) % (uint32_t)p.ny);
    const int z = (int)(n / ((uint32_t)p.nx * (uint32_t)p.ny));
    float drho = 0.f, jx = 0.f, jy = 0.f, jz = 0.f;
#pragma unroll
    for (int q = 0; q < 19; ++q) {
        const float h = natural_h<L>(p, state, q, n, x, y, z);
        drho += h;
        jx += (float)cx(q) * h;
        jy += (float)cy(q) * h;
        jz += (float)cz(q) * h;
    }
    const float r = 1.0f + drho;
    rho[k] = r;
    u0[k] = jx / r + 0.5f * p.g[0];
    u1[k] = jy / r + 0.5f * p.g[1];
    u2[k] = jz / r + 0.5f * p.g[2];
}

// The INLET cells' post-collision slots of a buffer in state `state` (ST_POST_AA: (opposite(q), s);
// ST_POST_AB: (q, s)) refilled with the reservoir's f_eq(rho_in, u_in) -- after a change of the
// flags or of the inlet state between steps, so that the next step's pulls read the new values
// (every step kernel keeps them there afterwards).
template <int L>
__global__ void __launch_bounds__(256) k_fill_inlet(Params p, int state) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= p.nx || y >= p.ny) return;
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    if ((p.flags[n] & TYPE_MASK) != T_INLET) return;
#pragma unroll
    for (int q = 0; q < 19; ++q)
        st<L>(p.A, idx<L>(state == ST_POST_AA ? opp(q) : q, n, p.N), p.heq_in[q]);
}

// ---- slab halos (A-B post-collision state, stored elements copied as they are) ------------------
// The five populations with c_z = sgn, k-th in q order, of plane z: buf[k * nx ny + x + nx y].
template <int L>
using Stored = typename std::conditional<L == LAYOUT_STREAM_FP16, __half, float>::type;

template <int L>
__global__ void __launch_bounds__(256) k_halo_pack(Params p, int z_lo, int z_hi, Stored<L>* lo,
                                                   Stored<L>* hi) {
    const size_t area = (size_t)p.nx * p.ny;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 10 * area) return;
    const bool up = i >= 5 * area;
    const size_t j = up ? i - 5 * area : i;
    const int k = (int)(j / area);
    const uint32_t xy = (uint32_t)(j - (size_t)k * area);
    const int q = face_velocity(2, up ? 1 : -1, k);
    const uint32_t n = xy + (uint32_t)area * (uint32_t)(up ? z_hi : z_lo);
    const Stored<L>* A = static_cast<const Stored<L>*>(p.A);
    (up ? hi : lo)[j] = A[idx_rt<L>(q, n, p.N)];
}

template <int L>
__global__ void __launch_bounds__(256) k_halo_unpack(Params p, const Stored<L>* below,
                                                     const Stored<L>* above) {
    const size_t area = (size_t)p.nx * p.ny;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 10 * area) return;
    const bool top = i >= 5 * area;  // the upper ghost plane takes the slab above's c_z = -1 values
    const size_t j = top ? i - 5 * area : i;
    const int k = (int)(j / area);
    const uint32_t xy = (uint32_t)(j - (size_t)k * area);
    const int q = face_velocity(2, top ? -1 : 1, k);
    const uint32_t n = xy + (uint32_t)area * (uint32_t)(top ? p.nz - 1 : 0);
    Stored<L>* A = static_cast<Stored<L>*>(p.A);
    A[idx_rt<L>(q, n, p.N)] = (top ? above : below)[j];
}

// Sets *bad when any stored population of a FLUID cell is not finite.
template <int L>
__global__ void __launch_bounds__(256) k_check_finite(Params p, int* bad) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= p.nx || y >= p.ny) return;
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    if ((p.flags[n] & TYPE_MASK) != T_FLUID) return;
    bool ok = true;
#pragma unroll
    for (int q = 0; q < 19; ++q) ok &= isfinite(ld<L>(p.A, idx<L>(q, n, p.N)));
    if (!ok) *bad = 1;
}

}  // namespace lbm
