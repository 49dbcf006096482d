// Boundary kernels of the AA odd and A-B pull steps: the special FLUID cells (a neighbour is a
// MOVING_WALL cell, or -- AA odd step -- a link crosses an OPEN face), one warp per cell.  Lane q < 19
// handles population q: it gathers it by the general per-link rules, the warp sums the moments,
// every lane relaxes its own population, and lane q scatters it (with the open-face copies and
// its link's momentum exchange).  A thread per cell walked the 19 links one after another, each
// waiting on a neighbour's flag byte and then on a population; here the 19 links are in flight
// together and there are 32 times as many threads for the few special cells of a grid.
//
// Per-link rules ("GPU lattice Boltzmann: streaming layout and performance", paragraph after the
// layout bullets; PortLBM §3.1; "GPU加速LBM流体仿真" §4.2): the source x - c_q is FLUID -> its
// post-collision value; SOLID -> x's own mirrored population; MOVING_WALL -> the mirrored one plus
// 6 w_q (c_q.u_w); INLET -> f_eq(rho_in, u_in); beyond an OPEN face -> the clamped cell's value
// (pre-gathered to scratch in the AA odd step).
#pragma once

#include "lbm_kernels.cuh"

namespace lbm {

constexpr int kSpecialCellsPerBlock = kWarpsPerBlock;  // 256 threads: 8 warps, 8 cells

// full-warp sum, the same value in every lane (lane 0's, broadcast)
__device__ __forceinline__ float warp_total(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return __shfl_sync(0xffffffffu, v, 0);
}
__device__ __forceinline__ float signed_by(int c, float v) { return c > 0 ? v : c < 0 ? -v : 0.0f; }

// Relaxation of population q (lane) given the cell's moments: the one-cell collision's formula.
template <bool BODY>
__device__ __forceinline__ float relax_lane(const Params& p, int q, int qx, int qy, int qz, float v) {
    const float drho = warp_total(v);
    const float jx = warp_total(signed_by(qx, v));
    const float jy = warp_total(signed_by(qy, v));
    const float jz = warp_total(signed_by(qz, v));
    const float rho = __fadd_rn(1.0f, drho);
    float inv = __frcp_rn(rho);
    asm("" : "+f"(inv));
    float ux, uy, uz;
    if (BODY) {
        ux = __fmaf_rn(jx, inv, p.tau_g[0]);
        uy = __fmaf_rn(jy, inv, p.tau_g[1]);
        uz = __fmaf_rn(jz, inv, p.tau_g[2]);
    } else {
        ux = __fmul_rn(jx, inv);
        uy = __fmul_rn(jy, inv);
        uz = __fmul_rn(jz, inv);
    }
    const float nuu15 = __fmul_rn(-1.5f, __fmaf_rn(ux, ux, __fmaf_rn(uy, uy, __fmul_rn(uz, uz))));
    const float cu = __fadd_rn(__fadd_rn(signed_by(qx, ux), signed_by(qy, uy)), signed_by(qz, uz));
    const float poly = q == 0 ? nuu15 : __fmaf_rn(cu, __fmaf_rn(4.5f, cu, 3.0f), nuu15);
    const float d = __fmaf_rn(-wq_rt(q), __fmaf_rn(rho, poly, drho), v);
    float hn = __fmaf_rn(-p.omega, d, v);
    if (BODY) hn = __fmaf_rn(rho, p.wk[q], hn);
    return hn;
}

// Momentum exchange of link q of a special cell (target type t of x + c_q, wrapped or clamped):
// SOLID gives 2 c_q f*_q, MOVING_WALL c_q (2 f*_q - 6 w_q (c_q.u_w)).
__device__ __forceinline__ void link_force(const Params& p, int q, int qx, int qy, int qz, int t,
                                           float hn, float& fx, float& fy, float& fz) {
    if (q == 0 || (t != T_SOLID && t != T_MOVING)) return;
    float f = 2.0f * (hn + wq_rt(q));
    if (t == T_MOVING) f -= p.wterm[q];
    fx += signed_by(qx, f);
    fy += signed_by(qy, f);
    fz += signed_by(qz, f);
}

// Cell of the special list handled by this warp; false past the end (warp-uniform).
__device__ __forceinline__ bool special_warp_cell(const Params& p, CellCoord& c) {
    const uint32_t i = blockIdx.x * kSpecialCellsPerBlock + (threadIdx.x >> 5);
    if (i >= p.n_special) return false;
    c.n = p.special[i];
    c.x = (int)(c.n % (uint32_t)p.nx);
    c.y = (int)((c.n / (uint32_t)p.nx) % (uint32_t)p.ny);
    c.z = (int)(c.n / ((uint32_t)p.nx * (uint32_t)p.ny));
    return true;
}

// AA odd step: the clamped cell's post-collision population written to the neighbours that take
// it as their source across an OPEN face (the zero-gradient outlet), population q of cell x.
template <int L>
__device__ __forceinline__ void face_copies_rt(const Params& p, int q, float v, int x, int y, int z) {
    const int c[3] = {cx_rt(q), cy_rt(q), cz_rt(q)};
    const int at[3] = {x, y, z};
    const int nn[3] = {p.nx, p.ny, p.nz};
    // axes on which x sits on the layer where c_q points into the domain from an OPEN face
    int M = 0;
    for (int a = 0; a < 3; ++a)
        if (c[a] != 0 && p.open[a] && ((c[a] > 0 && at[a] == 0) || (c[a] < 0 && at[a] == nn[a] - 1)))
            M |= 1 << a;
    if (M == 0) return;
    for (int S = 1; S < 8; ++S) {
        if ((S & M) != S) continue;
        // receiver r: on axes in S it shares x's coordinate (its source clamps back onto x)
        int r[3] = {x, y, z};
        bool valid = true;
        for (int a = 0; a < 3; ++a) {
            if (S & (1 << a)) continue;
            int v2 = r[a] + c[a];
            if (v2 < 0 || v2 >= nn[a]) {
                if (p.open[a]) valid = false;
                else v2 = v2 < 0 ? v2 + nn[a] : v2 - nn[a];
            }
            r[a] = v2;
        }
        if (!valid) continue;
        const uint32_t rc = (uint32_t)r[0] + (uint32_t)p.nx * ((uint32_t)r[1] + (uint32_t)p.ny * r[2]);
        if ((p.flags[rc] & TYPE_MASK) == T_FLUID) st<L>(p.A, idx_rt<L>(q, rc, p.N), v);
    }
}

// Boundary kernel of the AA odd step (gather: population q of x at (opposite(q), x - c_q);
// scatter: to (q, x + c_q); solid-type partners use x's own mirrored slots).
template <int L, bool FORCE, bool BODY>
__global__ void __launch_bounds__(256) k_aa_odd_special(Params p) {
    CellCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (special_warp_cell(p, c)) {
        const int lane = threadIdx.x & 31;
        const bool on = lane < 19;
        const int q = on ? lane : 0;
        const int qx = cx_rt(q), qy = cy_rt(q), qz = cz_rt(q);
        float v = 0.f;
        Link s{0u, -1};
        int ts = T_FLUID;
        if (on) {
            s = link_cell(p, c.x, c.y, c.z, -qx, -qy, -qz);
            const int t = ts = p.flags[s.cell] & TYPE_MASK;
            if (t == T_SOLID || t == T_MOVING) {
                v = ld<L>(p.A, idx_rt<L>(q, c.n, p.N));  // f*_opp(q)(x) sits at (q, x)
                if (t == T_MOVING) v += p.wterm[q];
            } else if (t == T_INLET) {
                v = p.heq_in[q];
            } else if (s.face >= 0) {
                v = p.scratch[scratch_slot(p, s.face, q, c.x, c.y, c.z)];
            } else {
                v = ld<L>(p.A, idx_rt<L>(opp_rt(q), s.cell, p.N));
            }
        }
        const float hn = relax_lane<BODY>(p, q, qx, qy, qz, v);
        // x + c_q is x - c_opp(q): lane opposite(q) already resolved that link and its type
        const int o = opp_rt(q);
        Link d;
        d.cell = __shfl_sync(0xffffffffu, s.cell, o);
        d.face = __shfl_sync(0xffffffffu, s.face, o);
        const int td = __shfl_sync(0xffffffffu, ts, o);
        if (on) {
            const int t = td;
            if (t == T_SOLID) {
                st<L>(p.A, idx_rt<L>(o, c.n, p.N), hn);                 // bounces back into x
            } else if (t == T_MOVING) {
                st<L>(p.A, idx_rt<L>(o, c.n, p.N), hn + p.wterm[o]);    // off the moving wall
            } else if (t == T_INLET) {
                // the reservoir feeds x: a direct INLET neighbour writes (o, x) itself (it is a
                // producer in the main kernel); one reached through an OPEN-face clamp does not
                if (d.face >= 0) st<L>(p.A, idx_rt<L>(o, c.n, p.N), p.heq_in[o]);
            } else if (d.face < 0) {
                st<L>(p.A, idx_rt<L>(q, d.cell, p.N), hn);
            }
            if (p.open[0] | p.open[1] | p.open[2]) face_copies_rt<L>(p, q, hn, c.x, c.y, c.z);
            if (FORCE) link_force(p, q, qx, qy, qz, t, hn, fx, fy, fz);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_special);
}

// Boundary kernel of the A-B pull: population q of x from (q, x - c_q) of A (the clamped cell
// beyond an OPEN face), collide, write (q, x) of B.
template <int L, bool FORCE, bool BODY>
__global__ void __launch_bounds__(256) k_ab_special(Params p) {
    CellCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (special_warp_cell(p, c)) {
        const int lane = threadIdx.x & 31;
        const bool on = lane < 19;
        const int q = on ? lane : 0;
        const int qx = cx_rt(q), qy = cy_rt(q), qz = cz_rt(q);
        float v = 0.f;
        int ts = T_FLUID;
        if (on) {
            const Link s = link_cell(p, c.x, c.y, c.z, -qx, -qy, -qz);
            const int t = ts = p.flags[s.cell] & TYPE_MASK;
            if (t == T_SOLID || t == T_MOVING) {
                v = ld<L>(p.A, idx_rt<L>(opp_rt(q), c.n, p.N));
                if (t == T_MOVING) v += p.wterm[q];
            } else if (t == T_INLET) {
                v = p.heq_in[q];
            } else {
                v = ld<L>(p.A, idx_rt<L>(q, s.cell, p.N));
            }
        }
        const float hn = relax_lane<BODY>(p, q, qx, qy, qz, v);
        // type of x + c_q = x - c_opp(q), resolved by lane opposite(q)
        const int td = __shfl_sync(0xffffffffu, ts, opp_rt(q));
        if (on) {
            st<L>(p.B, idx_rt<L>(q, c.n, p.N), hn);
            if (FORCE) link_force(p, q, qx, qy, qz, td, hn, fx, fy, fz);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_special);
}

}  // namespace lbm
