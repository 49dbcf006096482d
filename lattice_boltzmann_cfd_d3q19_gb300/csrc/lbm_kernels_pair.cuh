// Two-cell kernels of the hot steps, for the stream layouts (fp32 and fp16 storage) on grids with
// an even nx and 19 N <= 2^32.  A thread owns the x-adjacent cells a = (x, y, z), x even, and
// b = (x + 1, y, z); a is the even element of every population plane, so the pair's own slots,
// and every slot reached along a velocity with c_x = 0, are one aligned two-element word.  The
// collision of both cells runs in packed fp32x2 arithmetic (collide2) with bit-for-bit the
// results of the one-cell kernels, and each address computation serves both cells, which halves
// the instructions per cell update of the one-cell kernels (they are issue-bound in fp16 storage
// and in porous media).
//
// Same steps and per-link rules as the one-cell kernels ("GPU lattice Boltzmann: streaming layout
// and performance", "In place" and "Two buffers"), with one difference in which slots a launch
// touches, confined to slots that nothing reads: the even AA step and the A-B steps store both
// cells of a pair, so a non-FLUID cell beside a FLUID one gets its (never-read) slots overwritten,
// and in the A-B pull a special cell's destination slots are written before its boundary kernel
// overwrites them; the odd AA step also writes a bounced population to its neighbour slot, which
// belongs to the SOLID cell it bounced from and is read by nobody.  Otherwise the odd AA step
// stores per cell (a SOLID or special cell's stores would land in slots other cells read, and its
// boundary kernel runs at the same time).
#pragma once

#include <type_traits>

#include "lbm_kernels.cuh"

namespace lbm {

template <int L>
using Elem = typename std::conditional<L == LAYOUT_STREAM_FP16, __half, float>::type;

// one element / two adjacent elements (the first at an even offset) of a population buffer
template <int L>
__device__ __forceinline__ float ld1(const Elem<L>* e) {
    if constexpr (L == LAYOUT_STREAM_FP16) return __half2float(*e);
    else return *e;
}
template <int L>
__device__ __forceinline__ void st1(Elem<L>* e, float v) {
    if constexpr (L == LAYOUT_STREAM_FP16) *e = __float2half_rn(v);
    else *e = v;
}
template <int L>
__device__ __forceinline__ float2 ld2(const Elem<L>* e) {
    if constexpr (L == LAYOUT_STREAM_FP16) return __half22float2(*reinterpret_cast<const __half2*>(e));
    else return *reinterpret_cast<const float2*>(e);
}
template <int L>
__device__ __forceinline__ void st2(Elem<L>* e, float2 v) {
    if constexpr (L == LAYOUT_STREAM_FP16) *reinterpret_cast<__half2*>(e) = __float22half2_rn(v);
    else *reinterpret_cast<float2*>(e) = v;
}

// Stores of the odd AA step, with the evict-first ("streaming") cache hint in fp32 storage: the
// slots it writes are not read again in the step (measured: porous 512^3 odd step 3.74 -> 3.68 ms;
// the even step keeps plain stores, whose lines the next step reads from L2 on grids near its size).
template <int L>
__device__ __forceinline__ void st1s(Elem<L>* e, float v) {
    if constexpr (L == LAYOUT_STREAM_FP16) *e = __float2half_rn(v);
    else __stcs(e, v);
}
template <int L>
__device__ __forceinline__ void st2s(Elem<L>* e, float2 v) {
    if constexpr (L == LAYOUT_STREAM_FP16) *reinterpret_cast<__half2*>(e) = __float22half2_rn(v);
    else __stcs(reinterpret_cast<float2*>(e), v);
}

// Half-precision storage: two cells' stored values kept as one packed register until used.
__device__ __forceinline__ __half2 ld2h(const __half* e) { return *reinterpret_cast<const __half2*>(e); }
__device__ __forceinline__ __half2 pack_h(__half a, __half b) { return __halves2half2(a, b); }

// Thread -> cell pair of the 3D launch (threads along x own pairs); false for the ragged tail.
struct PairCoord {
    int x, y, z;  // coordinates of the even cell a
    uint32_t n;   // index of a (even)
};
// PLANES: the plane from zbase / zstep (the A-B step kernel, which also runs over some planes)
template <bool PLANES = false>
__device__ __forceinline__ bool grid_pair(const Params& p, PairCoord& c) {
    c.x = 2 * (int)(blockIdx.x * blockDim.x + threadIdx.x);
    c.y = blockIdx.y * blockDim.y + threadIdx.y;
    if constexpr (PLANES) c.z = p.zbase + p.zstep * (int)blockIdx.z;
    else c.z = p.zrev ? p.nz - 1 - (int)blockIdx.z : (int)blockIdx.z;
    c.n = (uint32_t)c.x + (uint32_t)p.nx * ((uint32_t)c.y + (uint32_t)p.ny * c.z);
    return c.x < p.nx && c.y < p.ny;
}

// Neighbour geometry of a pair: the y and z parts of n + s c_q are shared by both cells; along x,
// a - 1 and b + 1 may leave the row, a + 1 = b and b - 1 = a never do.  Offsets wrap on PERIODIC
// axes; with `clamp` (the A-B pulls) they clamp onto the last layer on OPEN axes, the
// zero-gradient source of a pull.  The AA odd kernels wrap everywhere: cells whose links cross an
// OPEN face are special and store nothing there, and an INLET producer drops such links.  `clamp`
// is a constant at every call site.
struct NbrPair {
    int dy[3], dz[3];  // y and z deltas for c = -1, 0, +1
    int wa;            // (a - 1) - a along x
    int wb;            // (b + 1) - a along x
    __device__ __forceinline__ NbrPair(const Params& p, int x, int y, int z, bool clamp) {
        const int sy = p.nx, sz = p.nx * p.ny;
        dy[0] = edge_delta(y, p.ny, sy, clamp && p.open[1], -1);
        dy[1] = 0;
        dy[2] = edge_delta(y, p.ny, sy, clamp && p.open[1], 1);
        dz[0] = edge_delta(z, p.nz, sz, clamp && p.open[2], -1);
        dz[1] = 0;
        dz[2] = edge_delta(z, p.nz, sz, clamp && p.open[2], 1);
        wa = x == 0 ? (clamp && p.open[0] ? 0 : p.nx - 1) : -1;
        wb = x + 2 == p.nx ? (clamp && p.open[0] ? 1 : 2 - p.nx) : 2;
    }
    // a + (0, s cy(Q), s cz(Q)), before the x part
    template <int Q, int S>
    __device__ __forceinline__ uint32_t yz(uint32_t n) const {
        return n + (uint32_t)(dy[S * cy(Q) + 1] + dz[S * cz(Q) + 1]);
    }
    // element offsets (from the one of a + yz part) of the cells a + S c_Q and b + S c_Q
    template <int Q, int S>
    __device__ __forceinline__ int xa() const {
        constexpr int sx = S * cx(Q);
        return sx == 0 ? 0 : sx < 0 ? wa : 1;
    }
    template <int Q, int S>
    __device__ __forceinline__ int xb() const {
        constexpr int sx = S * cx(Q);
        return sx == 0 ? 1 : sx < 0 ? 0 : wb;
    }
    // the two cells a + S c_Q, b + S c_Q: element e of the plane holding (a + yz part) -> values
    template <int L, int Q, int S>
    __device__ __forceinline__ float2 load(const Elem<L>* e) const {
        constexpr int sx = S * cx(Q);
        if constexpr (sx == 0) return ld2<L>(e);
        else if constexpr (sx < 0) return make_float2(ld1<L>(e + wa), ld1<L>(e));
        else return make_float2(ld1<L>(e + 1), ld1<L>(e + wb));
    }
    // the same, half-precision storage, packed without conversion
    template <int Q, int S>
    __device__ __forceinline__ __half2 load_h(const __half* e) const {
        constexpr int sx = S * cx(Q);
        if constexpr (sx == 0) return ld2h(e);
        else if constexpr (sx < 0) return pack_h(e[wa], e[0]);
        else return pack_h(e[1], e[wb]);
    }
    template <int L, int Q, int S, bool BOTH>
    __device__ __forceinline__ void store(Elem<L>* e, float2 v, bool act_a, bool act_b) const {
        constexpr int sx = S * cx(Q);
        if constexpr (sx == 0) {
            if (BOTH) {
                st2s<L>(e, v);
            } else {
                if (act_a) st1s<L>(e, v.x);
                if (act_b) st1s<L>(e + 1, v.y);
            }
        } else if constexpr (sx < 0) {
            if (BOTH || act_a) st1s<L>(e + wa, v.x);
            if (BOTH || act_b) st1s<L>(e, v.y);
        } else {
            if (BOTH || act_a) st1s<L>(e + 1, v.x);
            if (BOTH || act_b) st1s<L>(e + wb, v.y);
        }
    }
};

// flag bytes and solid-link masks of a pair (both at an even index: one aligned load each)
struct PairFlags {
    uint8_t fa, fb;
    uint32_t ma, mb;
};
__device__ __forceinline__ PairFlags pair_flags(const Params& p, uint32_t n, bool want_mask) {
    PairFlags f;
    const uint16_t fl = *reinterpret_cast<const uint16_t*>(p.flags + n);
    f.fa = (uint8_t)(fl & 0xffu);
    f.fb = (uint8_t)(fl >> 8);
    if (want_mask) {
        const uint2 m = *reinterpret_cast<const uint2*>(p.mask + n);
        f.ma = m.x;
        f.mb = m.y;
    } else {
        f.ma = f.mb = 0u;
    }
    return f;
}

// INLET cells as producers ("PortLBM", §3.1, last paragraph: the inlet imposes the equilibrium):
// an INLET cell's post-collision state is the reservoir's f_eq(rho_in, u_in), stored by the step
// kernels where a FLUID cell's would be, so that its neighbours read it through the ordinary
// addressing.  The two-cell kernels do this in a tail pass after their main work, which re-reads
// the pair's flag word and recomputes its coordinates: nothing about inlets is held in registers
// through the collision and the scatter (the main path may have stored a value for the inlet cell
// of a mixed pair first; the tail pass, in the same thread, overwrites it).
__device__ __forceinline__ bool is_inlet(const Params& p, bool in, uint8_t f) {
    return in && p.any_inlet && (f & TYPE_MASK) == T_INLET;
}
template <bool PLANES = false>
__device__ __forceinline__ bool pair_inlets(const Params& p, PairCoord& c, bool& ia, bool& ib) {
    if (!p.any_inlet || !grid_pair<PLANES>(p, c)) return false;
    const uint16_t fl = *reinterpret_cast<const uint16_t*>(p.flags + c.n);
    ia = (fl & TYPE_MASK) == T_INLET;
    ib = ((fl >> 8) & TYPE_MASK) == T_INLET;
    return ia || ib;
}
// f_eq - w of the reservoir into the pair's slots of plane (OPP ? opposite(q) : q) of buf (the
// even AA step: opposite(q); the A-B steps: q of the destination)
template <int L, bool OPP>
__device__ __forceinline__ void pair_inlet_store(const Params& p, void* buf, uint32_t n, bool ia,
                                                 bool ib) {
    Elem<L>* B = static_cast<Elem<L>*>(buf);
#pragma unroll
    for (int q = 0; q < 19; ++q) {
        Elem<L>* e = B + (p.plane32[OPP ? opp(q) : q] + n);
        if (ia) st1<L>(e, p.heq_in[q]);
        if (ib) st1<L>(e + 1, p.heq_in[q]);
    }
}

// Momentum exchange of a pair, packed: the sum over the links q whose bit is set in the cell's
// mask of c_q f*_q, f* = h* + w (per cell, one lane each); twice that is the force the fluid
// gives up (bounce-back returns 2 c_q f*_q), so the factor 2 is applied once, in into().
struct PairForce {
    float2 x = make_float2(0.f, 0.f), y = make_float2(0.f, 0.f), z = make_float2(0.f, 0.f);
    template <int Q>
    __device__ __forceinline__ void link(float2 h_post, bool ba, bool bb) {
        const float2 hw = Arith2::add(h_post, Arith2::splat(wq(Q)));
        const float2 t = make_float2(ba ? hw.x : 0.f, bb ? hw.y : 0.f);
        if (cx(Q) > 0) x = Arith2::add(x, t); else if (cx(Q) < 0) x = Arith2::sub(x, t);
        if (cy(Q) > 0) y = Arith2::add(y, t); else if (cy(Q) < 0) y = Arith2::sub(y, t);
        if (cz(Q) > 0) z = Arith2::add(z, t); else if (cz(Q) < 0) z = Arith2::sub(z, t);
    }
    template <int Q = 1>
    __device__ __forceinline__ void masks(uint32_t ma, uint32_t mb, const float2 (&h)[19]) {
        link<Q>(h[Q], solid_link<Q>(ma), solid_link<Q>(mb));
        if constexpr (Q < 18) masks<Q + 1>(ma, mb, h);
    }
    // add to the thread's (one-cell convention) accumulators
    __device__ __forceinline__ void into(float& fx, float& fy, float& fz) const {
        fx += 2.0f * (x.x + x.y);
        fy += 2.0f * (y.x + y.y);
        fz += 2.0f * (z.x + z.y);
    }
};

// Gather of a pull (AA odd: FAR_OPP, population q from (opposite(q), x - c_q); A-B: from
// (q, x - c_q)).  WALL: a cell whose link opposite(q) is a solid link takes its own mirrored slot
// instead, (q, x) in AA and (opposite(q), x) in A-B; each cell then selects its address and
// loads one element (no branches: all 38 loads are independent).  Without WALL the pair's
// elements are loaded together where they are adjacent and aligned.
template <int L, bool FAR_OPP, bool WALL, int Q = 0>
__device__ __forceinline__ void pair_gather(const Params& p, const NbrPair& nb, uint32_t n,
                                            uint32_t ma, uint32_t mb, float2 (&h)[19]) {
    const Elem<L>* A = static_cast<const Elem<L>*>(p.A);
    constexpr int far_plane = FAR_OPP ? opp(Q) : Q;
    constexpr int own_plane = FAR_OPP ? Q : opp(Q);
    const uint32_t far = p.plane32[far_plane] + nb.template yz<Q, -1>(n);
    if constexpr (WALL && Q > 0) {
        const uint32_t own = p.plane32[own_plane] + n;
        const uint32_t oa = solid_link<opp(Q)>(ma) ? own : far + (uint32_t)nb.template xa<Q, -1>();
        const uint32_t ob = solid_link<opp(Q)>(mb) ? own + 1u : far + (uint32_t)nb.template xb<Q, -1>();
        h[Q] = make_float2(ld1<L>(A + oa), ld1<L>(A + ob));
    } else {
        h[Q] = nb.template load<L, Q, -1>(A + far);
    }
    if constexpr (Q < 18) pair_gather<L, FAR_OPP, WALL, Q + 1>(p, nb, n, ma, mb, h);
}

// The gather in half-precision storage: the same addresses as pair_gather, the values kept packed.
template <bool FAR_OPP, bool WALL, int Q = 0>
__device__ __forceinline__ void pair_gather_h(const Params& p, const NbrPair& nb, uint32_t n,
                                              uint32_t ma, uint32_t mb, __half2 (&hh)[19]) {
    const __half* A = static_cast<const __half*>(p.A);
    constexpr int far_plane = FAR_OPP ? opp(Q) : Q;
    constexpr int own_plane = FAR_OPP ? Q : opp(Q);
    const uint32_t far = p.plane32[far_plane] + nb.template yz<Q, -1>(n);
    if constexpr (WALL && Q > 0) {
        const uint32_t own = p.plane32[own_plane] + n;
        const uint32_t oa = solid_link<opp(Q)>(ma) ? own : far + (uint32_t)nb.template xa<Q, -1>();
        const uint32_t ob = solid_link<opp(Q)>(mb) ? own + 1u : far + (uint32_t)nb.template xb<Q, -1>();
        hh[Q] = pack_h(A[oa], A[ob]);
    } else {
        hh[Q] = nb.template load_h<Q, -1>(A + far);
    }
    if constexpr (Q < 18) pair_gather_h<FAR_OPP, WALL, Q + 1>(p, nb, n, ma, mb, hh);
}

// Half-precision storage: which kernels keep the stored pairs packed (fewer registers, 6 blocks
// per SM) and relax each population where it is stored.  Measured at 512^3: the even step gains
// (1.72 -> 1.60 ms); the odd and A-B steps, which also hold neighbour geometry, spilled at 5-6
// blocks and lost, and keep the fp32 arrays at 4 blocks (the A-B pull has no packed form).
constexpr bool kPackedHalfEven = true;
constexpr bool kPackedHalfOdd = false;
constexpr int kOddBlocksNoWalls = 4;
template <int L>
constexpr int pair_min_blocks(bool packed) { return L == LAYOUT_STREAM_FP16 && packed ? 6 : 4; }

// Post-collision values of a pair, population by population: an array relaxed in place (fp32
// storage), or the relaxation of the stored half-precision values, done where each is stored
// (the fp32 values of all 19 populations are then never held at once).
struct ArraySrc {
    const float2 (&h)[19];
    template <int Q>
    __device__ __forceinline__ float2 get() const { return h[Q]; }
};
template <bool BODY>
struct RelaxSrc {
    const Moments<Arith2>& m;
    const __half2 (&hh)[19];
    const Params& p;
    template <int Q>
    __device__ __forceinline__ float2 get() const {
        // a fresh conversion of the stored pair (opaque to the compiler, so the moments pass's
        // fp32 values are not kept alive for it)
        unsigned bits = *reinterpret_cast<const unsigned*>(&hh[Q]);
        asm volatile("" : "+r"(bits));
        return relax_q<Arith2, BODY>(m, Q, __half22float2(*reinterpret_cast<const __half2*>(&bits)), p);
    }
};

// Momentum exchange of the MOVING_WALL links of cell (x, y, z), population Q with post-collision
// value h: c_Q (2 f*_Q - 6 w_Q (c_Q.u_w)) when x + c_Q is a MOVING_WALL cell.
template <int Q>
__device__ __forceinline__ void moving_link(const Params& p, int x, int y, int z, float h, float& fx,
                                            float& fy, float& fz) {
    const Link d = link_cell(p, x, y, z, cx(Q), cy(Q), cz(Q));
    if ((p.flags[d.cell] & TYPE_MASK) == T_MOVING) {
        const float t = 2.0f * (h + wq(Q)) - p.wterm[Q];
        if (cx(Q) > 0) fx += t; else if (cx(Q) < 0) fx -= t;
        if (cy(Q) > 0) fy += t; else if (cy(Q) < 0) fy -= t;
        if (cz(Q) > 0) fz += t; else if (cz(Q) < 0) fz -= t;
    }
}

// Stores of a pair at its own slots (plane opposite(q) in the AA even step, plane q in the A-B
// steps), with the momentum exchange of the solid links (masks ma, mb) and of the moving-wall links
// (cells with mov_a / mov_b set).
template <int L, bool OPP_PLANE, bool FORCE, int Q = 0, typename S>
__device__ __forceinline__ void own_store(const Params& p, Elem<L>* base, uint32_t n, const S& src,
                                          uint32_t ma, uint32_t mb, bool mov_a, bool mov_b, int x,
                                          int y, int z, PairForce& pf, float& fx, float& fy,
                                          float& fz) {
    const float2 v = src.template get<Q>();
    st2<L>(base + (p.plane32[OPP_PLANE ? opp(Q) : Q] + n), v);
    if constexpr (FORCE && Q > 0) {
        pf.template link<Q>(v, solid_link<Q>(ma), solid_link<Q>(mb));
        if (mov_a) moving_link<Q>(p, x, y, z, v.x, fx, fy, fz);
        if (mov_b) moving_link<Q>(p, x + 1, y, z, v.y, fx, fy, fz);
    }
    if constexpr (Q < 18)
        own_store<L, OPP_PLANE, FORCE, Q + 1>(p, base, n, src, ma, mb, mov_a, mov_b, x, y, z, pf, fx, fy, fz);
}

// ============================== AA pattern, even step, two cells ================================
// Every FLUID cell; the pair's slots are read and written as aligned words.
// Resident blocks per SM: 4 for fp32 storage (64 registers), 6 for the packed half-precision form
// (40 registers); the fp16 kernel on fp32 arrays with 66 registers fell to 3 blocks and lost 9%.
// INLETS: the kernel carries the INLET tail pass (off only for a domain without inlets, in the
// half-precision instantiations: an issue-bound kernel pays for even a never-taken epilogue).
template <int L, bool FORCE, bool BODY, bool INLETS>
__global__ void __launch_bounds__(256, pair_min_blocks<L>(kPackedHalfEven)) k_aa_even2(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (grid_pair(p, c)) {
        const PairFlags f = pair_flags(p, c.n, false);
        const bool act_a = (f.fa & TYPE_MASK) == T_FLUID, act_b = (f.fb & TYPE_MASK) == T_FLUID;
        if ((act_a || act_b) && L == LAYOUT_STREAM_FP16 && kPackedHalfEven) {
            // half-precision storage: the stored pairs stay packed; each population is relaxed
            // where it is stored
            __half* A = static_cast<__half*>(p.A);
            __half2 hh[19];
#pragma unroll
            for (int q = 0; q < 19; ++q) hh[q] = ld2h(A + (p.plane32[q] + c.n));
            const Moments<Arith2> m = moments<Arith2, BODY>(HalfPairView{hh}, p);
            uint32_t ns = c.n;
            asm volatile("" : "+r"(ns) : "f"(m.rho.x), "f"(m.rho.y));
            uint32_t ma = 0u, mb = 0u;
            bool mov_a = false, mov_b = false;
            if (FORCE) {
                const bool wa_ = act_a && !(f.fa & F_BULK), wb_ = act_b && !(f.fb & F_BULK);
                if (wa_ || wb_) {
                    const uint2 mm = *reinterpret_cast<const uint2*>(p.mask + c.n);
                    ma = wa_ ? mm.x : 0u;
                    mb = wb_ ? mm.y : 0u;
                }
                mov_a = p.any_moving && wa_ && (f.fa & F_SPECIAL);
                mov_b = p.any_moving && wb_ && (f.fb & F_SPECIAL);
            }
            PairForce pf;
            own_store<L, true, FORCE>(p, reinterpret_cast<Elem<L>*>(A), ns, RelaxSrc<BODY>{m, hh, p},
                                      ma, mb, mov_a, mov_b, c.x, c.y, c.z, pf, fx, fy, fz);
            if (FORCE) pf.into(fx, fy, fz);
        } else if (act_a || act_b) {
            Elem<L>* A = static_cast<Elem<L>*>(p.A);
            float2 h[19];
#pragma unroll
            for (int q = 0; q < 19; ++q) h[q] = ld2<L>(A + (p.plane32[q] + c.n));
            collide2<BODY>(h, p);
            uint32_t ns = c.n;
            asm volatile("" : "+r"(ns) : "f"(h[0].x), "f"(h[18].y));
#pragma unroll
            for (int q = 0; q < 19; ++q) st2<L>(A + (p.plane32[opp(q)] + ns), h[q]);
            if (FORCE) {
                const bool wa_ = act_a && !(f.fa & F_BULK), wb_ = act_b && !(f.fb & F_BULK);
                if (wa_ || wb_) {
                    const uint2 m = *reinterpret_cast<const uint2*>(p.mask + c.n);
                    PairForce pf;
                    pf.masks(wa_ ? m.x : 0u, wb_ ? m.y : 0u, h);
                    pf.into(fx, fy, fz);
                    if (p.any_moving) {
                        if (wa_ && (f.fa & F_SPECIAL))
                            moving_forces(p, PairLane<0>{h}, c.x, c.y, c.z, fx, fy, fz);
                        if (wb_ && (f.fb & F_SPECIAL))
                            moving_forces(p, PairLane<1>{h}, c.x + 1, c.y, c.z, fx, fy, fz);
                    }
                }
            }
        }
    }
    if constexpr (INLETS) {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets(p, ci, ia, ib)) pair_inlet_store<L, true>(p, p.A, ci.n, ia, ib);
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// ============================== AA pattern, even step, bundle layout, two cells =================
// The bundle layout ([PortLBM] Fig. 2(c): the populations sharing (c_y, c_z) form a bundle, a
// cell's members of one bundle stored together) on an even nx: a pair's records of one bundle are
// one run of 2 m elements (m = 3 or 1 members) starting at an even element, so the 19 populations
// of both cells load and store as 19 aligned two-element words, as in the stream layout (element
// accesses at the bundle's stride touched 3 times the sectors per request).

// member j (c_x = j - 1) of the bundle whose first member is q0; the only member of a 1-bundle
__host__ __device__ constexpr int bundle_member(int q0, int j) {
    for (int q = 0; q < 19; ++q)
        if (cy(q) == cy(q0) && cz(q) == cz(q0) && (bundle_size(q0) == 1 || cx(q) == j - 1)) return q;
    return -1;
}

// the pair's populations of the bundle that starts at Q (bundle_j(Q) == 0), then the next bundles
template <int Q = 0>
__device__ __forceinline__ void bundle_gather2(const float* A, uint32_t N, uint32_t a, float2 (&h)[19]) {
    if constexpr (bundle_j(Q) == 0) {
        const float* e = A + ((uint32_t)bundle_off(Q) * N + a * (uint32_t)bundle_size(Q));
        if constexpr (bundle_size(Q) == 3) {
            // [a0 a1 a2 b0 b1 b2] as three words
            const float2 w0 = ld2<LAYOUT_BUNDLE>(e), w1 = ld2<LAYOUT_BUNDLE>(e + 2),
                         w2 = ld2<LAYOUT_BUNDLE>(e + 4);
            h[bundle_member(Q, 0)] = make_float2(w0.x, w1.y);
            h[bundle_member(Q, 1)] = make_float2(w0.y, w2.x);
            h[bundle_member(Q, 2)] = make_float2(w1.x, w2.y);
        } else {
            h[Q] = ld2<LAYOUT_BUNDLE>(e);
        }
    }
    if constexpr (Q < 18) bundle_gather2<Q + 1>(A, N, a, h);
}

// AA even store: member p of a bundle receives the collided population opposite(p)
template <int Q = 0>
__device__ __forceinline__ void bundle_scatter2_opp(float* A, uint32_t N, uint32_t a,
                                                    const float2 (&h)[19]) {
    if constexpr (bundle_j(Q) == 0) {
        float* e = A + ((uint32_t)bundle_off(Q) * N + a * (uint32_t)bundle_size(Q));
        if constexpr (bundle_size(Q) == 3) {
            const float2 v0 = h[opp(bundle_member(Q, 0))], v1 = h[opp(bundle_member(Q, 1))],
                         v2 = h[opp(bundle_member(Q, 2))];
            st2<LAYOUT_BUNDLE>(e, make_float2(v0.x, v1.x));
            st2<LAYOUT_BUNDLE>(e + 2, make_float2(v2.x, v0.y));
            st2<LAYOUT_BUNDLE>(e + 4, make_float2(v1.y, v2.y));
        } else {
            st2<LAYOUT_BUNDLE>(e, h[opp(Q)]);
        }
    }
    if constexpr (Q < 18) bundle_scatter2_opp<Q + 1>(A, N, a, h);
}

template <bool FORCE, bool BODY>
__global__ void __launch_bounds__(256, 4) k_aa_even2_bundle(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (grid_pair(p, c)) {
        const PairFlags f = pair_flags(p, c.n, false);
        const bool act_a = (f.fa & TYPE_MASK) == T_FLUID, act_b = (f.fb & TYPE_MASK) == T_FLUID;
        if (act_a || act_b) {
            float* A = static_cast<float*>(p.A);
            const uint32_t N = (uint32_t)p.N;
            float2 h[19];
            bundle_gather2(A, N, c.n, h);
            collide2<BODY>(h, p);
            uint32_t ns = c.n;
            asm volatile("" : "+r"(ns) : "f"(h[0].x), "f"(h[18].y));
            bundle_scatter2_opp(A, N, ns, h);
            if (FORCE) {
                const bool wa_ = act_a && !(f.fa & F_BULK), wb_ = act_b && !(f.fb & F_BULK);
                if (wa_ || wb_) {
                    const uint2 m = *reinterpret_cast<const uint2*>(p.mask + c.n);
                    PairForce pf;
                    pf.masks(wa_ ? m.x : 0u, wb_ ? m.y : 0u, h);
                    pf.into(fx, fy, fz);
                    if (p.any_moving) {
                        if (wa_ && (f.fa & F_SPECIAL))
                            moving_forces(p, PairLane<0>{h}, c.x, c.y, c.z, fx, fy, fz);
                        if (wb_ && (f.fb & F_SPECIAL))
                            moving_forces(p, PairLane<1>{h}, c.x + 1, c.y, c.z, fx, fy, fz);
                    }
                }
            }
        }
    }
    {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets(p, ci, ia, ib)) {
#pragma unroll
            for (int q = 0; q < 19; ++q) {
                if (ia) st<LAYOUT_BUNDLE>(p.A, idx<LAYOUT_BUNDLE, uint32_t>(opp(q), ci.n, (uint32_t)p.N), p.heq_in[q]);
                if (ib) st<LAYOUT_BUNDLE>(p.A, idx<LAYOUT_BUNDLE, uint32_t>(opp(q), ci.n + 1, (uint32_t)p.N), p.heq_in[q]);
            }
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// ============================== AA pattern, odd step, bundle layout, two cells ===================
// The AA odd step in the bundle layout on an even nx.  Population q, member m = c_x + 1 of bundle
// (c_y, c_z), comes from member 2 - m of the opposite bundle in the record of x - c_q and goes to
// member m of its own bundle in the record of x + c_q.  For a pair (a = x, b = x + 1) the six
// elements one bundle of three members touches on one row lie in the records x - 1 .. x + 2: two
// aligned words inside the pair's own two records (e .. e + 1 and e + 4 .. e + 5, e = 3 x
// relative to the row) and one element on either side.  A bundle of one member is one aligned
// word, as in the stream layout.  Element by element, each of those accesses touched a third of
// the sectors of a request.  Warps with a solid link select each cell's own mirrored slot per
// element, as the stream-layout kernel does.  3 blocks per SM (80 registers): at 4 (64 registers)
// the kernel spilled and took 0.468 ms at 256^3 instead of 0.427.

// element offset of population q of cell n in the bundle layout
template <int Q>
__device__ __forceinline__ uint32_t bidx(uint32_t N, uint32_t n) {
    return idx<LAYOUT_BUNDLE, uint32_t>(Q, n, N);
}
// the solid-link select of the gather: own mirrored slot (q, x) when the link opposite(q) is solid
template <int Q>
__device__ __forceinline__ uint32_t bsel(uint32_t m, uint32_t own, uint32_t far) {
    if constexpr (Q == 0) return far;
    else return solid_link<opp(Q)>(m) ? own : far;
}

// the own mirrored slot (opposite(q), x) of a cell whose link q is solid, and the link's momentum
// exchange
template <int Q, bool FORCE>
__device__ __forceinline__ void bundle_bounce(float* A, uint32_t N, uint32_t n, uint32_t ma,
                                              uint32_t mb, float2 v, PairForce& pf) {
    const bool ba = solid_link<Q>(ma), bb = solid_link<Q>(mb);
    if (ba) st1s<LAYOUT_BUNDLE>(A + bidx<opp(Q)>(N, n), v.x);
    if (bb) st1s<LAYOUT_BUNDLE>(A + bidx<opp(Q)>(N, n + 1), v.y);
    if (FORCE) pf.template link<Q>(v, ba, bb);
}

template <bool WALL, int Q = 0>
__device__ __forceinline__ void bundle_odd_gather2(const float* A, uint32_t N, const NbrPair& nb,
                                                   uint32_t n, uint32_t ma, uint32_t mb,
                                                   float2 (&h)[19]) {
    if constexpr (bundle_j(Q) == 0) {
        // the source: the opposite bundle on the row (y - c_y, z - c_z)
        const uint32_t r = nb.template yz<Q, -1>(n);
        if constexpr (bundle_size(Q) == 3) {
            constexpr int m0 = bundle_member(Q, 0), m1 = bundle_member(Q, 1), m2 = bundle_member(Q, 2);
            const uint32_t e = (uint32_t)bundle_off(opp(Q)) * N + 3u * r;
            if constexpr (WALL) {
                h[m2] = make_float2(A[bsel<m2>(ma, bidx<m2>(N, n), e + 3 * nb.wa)],
                                    A[bsel<m2>(mb, bidx<m2>(N, n + 1), e)]);
                h[m1] = make_float2(A[bsel<m1>(ma, bidx<m1>(N, n), e + 1)],
                                    A[bsel<m1>(mb, bidx<m1>(N, n + 1), e + 4)]);
                h[m0] = make_float2(A[bsel<m0>(ma, bidx<m0>(N, n), e + 5)],
                                    A[bsel<m0>(mb, bidx<m0>(N, n + 1), e + 3 * nb.wb + 2)]);
            } else {
                const float2 w0 = ld2<LAYOUT_BUNDLE>(A + e), w1 = ld2<LAYOUT_BUNDLE>(A + e + 4);
                h[m2] = make_float2(A[e + 3 * nb.wa], w0.x);
                h[m1] = make_float2(w0.y, w1.x);
                h[m0] = make_float2(w1.y, A[e + 3 * nb.wb + 2]);
            }
        } else {
            const uint32_t e = (uint32_t)bundle_off(opp(Q)) * N + r;
            if constexpr (WALL)
                h[Q] = make_float2(A[bsel<Q>(ma, bidx<Q>(N, n), e)],
                                   A[bsel<Q>(mb, bidx<Q>(N, n + 1), e + 1)]);
            else
                h[Q] = ld2<LAYOUT_BUNDLE>(A + e);
        }
    }
    if constexpr (Q < 18) bundle_odd_gather2<WALL, Q + 1>(A, N, nb, n, ma, mb, h);
}

// the scatter: the pair's slots in the records of x + c_q (whole words when both cells work,
// else per cell), and with WALL on each solid link also the own mirrored slot (opposite(q), x)
// and the link's momentum exchange
template <bool WALL, bool BOTH, bool FORCE, int Q = 0>
__device__ __forceinline__ void bundle_odd_scatter2(float* A, uint32_t N, const NbrPair& nb,
                                                    uint32_t n, uint32_t ma, uint32_t mb,
                                                    bool act_a, bool act_b, const float2 (&h)[19],
                                                    PairForce& pf) {
    if constexpr (bundle_j(Q) == 0) {
        // the destination: this bundle on the row (y + c_y, z + c_z)
        const uint32_t r = nb.template yz<Q, 1>(n);
        if constexpr (bundle_size(Q) == 3) {
            constexpr int m0 = bundle_member(Q, 0), m1 = bundle_member(Q, 1), m2 = bundle_member(Q, 2);
            const uint32_t e = (uint32_t)bundle_off(Q) * N + 3u * r;
            const float2 v0 = h[m0], v1 = h[m1], v2 = h[m2];
            if constexpr (BOTH) {
                st2s<LAYOUT_BUNDLE>(A + e, make_float2(v0.y, v1.x));
                st2s<LAYOUT_BUNDLE>(A + e + 4, make_float2(v1.y, v2.x));
                st1s<LAYOUT_BUNDLE>(A + e + 3 * nb.wa, v0.x);
                st1s<LAYOUT_BUNDLE>(A + e + 3 * nb.wb + 2, v2.y);
            } else {
                if (act_a) {
                    st1s<LAYOUT_BUNDLE>(A + e + 3 * nb.wa, v0.x);
                    st1s<LAYOUT_BUNDLE>(A + e + 1, v1.x);
                    st1s<LAYOUT_BUNDLE>(A + e + 5, v2.x);
                }
                if (act_b) {
                    st1s<LAYOUT_BUNDLE>(A + e, v0.y);
                    st1s<LAYOUT_BUNDLE>(A + e + 4, v1.y);
                    st1s<LAYOUT_BUNDLE>(A + e + 3 * nb.wb + 2, v2.y);
                }
            }
            if constexpr (WALL) {
                bundle_bounce<m0, FORCE>(A, N, n, ma, mb, v0, pf);
                if constexpr (m1 != 0) bundle_bounce<m1, FORCE>(A, N, n, ma, mb, v1, pf);
                bundle_bounce<m2, FORCE>(A, N, n, ma, mb, v2, pf);
            }
        } else {
            const uint32_t e = (uint32_t)bundle_off(Q) * N + r;
            if constexpr (BOTH) {
                st2s<LAYOUT_BUNDLE>(A + e, h[Q]);
            } else {
                if (act_a) st1s<LAYOUT_BUNDLE>(A + e, h[Q].x);
                if (act_b) st1s<LAYOUT_BUNDLE>(A + e + 1, h[Q].y);
            }
            if constexpr (WALL) bundle_bounce<Q, FORCE>(A, N, n, ma, mb, h[Q], pf);
        }
    }
    if constexpr (Q < 18)
        bundle_odd_scatter2<WALL, BOTH, FORCE, Q + 1>(A, N, nb, n, ma, mb, act_a, act_b, h, pf);
}

// INLET producers of the odd step in the bundle layout: f_eq,q of the reservoir to (q, s + c_q),
// links leaving through an OPEN face dropped (as odd2_produce)
template <int Q = 1>
__device__ __forceinline__ void odd2_produce_bundle(const Params& p, const NbrPair& nb, uint32_t n,
                                                    int x, int y, int z, bool ia, bool ib) {
    float* A = static_cast<float*>(p.A);
    const uint32_t N = (uint32_t)p.N;
    const uint32_t r = nb.template yz<Q, 1>(n);
    const bool yz_out = (cy(Q) != 0 && p.open[1] && y == (cy(Q) > 0 ? p.ny - 1 : 0)) ||
                        (cz(Q) != 0 && p.open[2] && z == (cz(Q) > 0 ? p.nz - 1 : 0));
    const bool xa_out = cx(Q) < 0 && p.open[0] && x == 0;
    const bool xb_out = cx(Q) > 0 && p.open[0] && x + 2 == p.nx;
    if (ia && !yz_out && !xa_out) A[bidx<Q>(N, r + (uint32_t)nb.template xa<Q, 1>())] = p.heq_in[Q];
    if (ib && !yz_out && !xb_out) A[bidx<Q>(N, r + (uint32_t)nb.template xb<Q, 1>())] = p.heq_in[Q];
    if constexpr (Q < 18) odd2_produce_bundle<Q + 1>(p, nb, n, x, y, z, ia, ib);
}

// WALLS = false: the grid has no solid link (the near-wall gather and scatter compiled out:
// periodic 256^3 0.427 -> 0.402 ms at the same 3 blocks per SM; at 4 it spilled, 0.447)
template <bool FORCE, bool BODY, bool INLETS, bool WALLS = true>
__global__ void __launch_bounds__(256, 3) k_aa_odd2_bundle(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const bool in = grid_pair(p, c);
    PairFlags f{0, 0, 0u, 0u};
    if (in) f = pair_flags(p, c.n, WALLS && p.any_solid_link != 0);
    const bool act_a = in && (f.fa & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
    const bool act_b = in && (f.fb & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
    if (!act_a) f.ma = 0u;
    if (!act_b) f.mb = 0u;
    const bool wall = WALLS && __any_sync(0xffffffffu, (f.ma | f.mb) != 0u);
    const bool both = __all_sync(0xffffffffu, act_a == act_b);
    if (act_a || act_b) {
        float* A = static_cast<float*>(p.A);
        const uint32_t N = (uint32_t)p.N;
        float2 h[19];
        {
            const NbrPair nb(p, c.x, c.y, c.z, false);
            if (wall) bundle_odd_gather2<true>(A, N, nb, c.n, f.ma, f.mb, h);
            else bundle_odd_gather2<false>(A, N, nb, c.n, f.ma, f.mb, h);
        }
        collide2<BODY>(h, p);
        uint32_t ns = c.n, mas = f.ma, mbs = f.mb;
        int xs = c.x, ys = c.y, zs = c.z;
        asm volatile("" : "+r"(ns), "+r"(mas), "+r"(mbs), "+r"(xs), "+r"(ys), "+r"(zs)
                     : "f"(h[0].x), "f"(h[18].y));
        const NbrPair nb(p, xs, ys, zs, false);
        PairForce pf;
        if (wall) {
            if (both) bundle_odd_scatter2<true, true, FORCE>(A, N, nb, ns, mas, mbs, act_a, act_b, h, pf);
            else bundle_odd_scatter2<true, false, FORCE>(A, N, nb, ns, mas, mbs, act_a, act_b, h, pf);
            if (FORCE) pf.into(fx, fy, fz);
        } else {
            if (both) bundle_odd_scatter2<false, true, FORCE>(A, N, nb, ns, mas, mbs, act_a, act_b, h, pf);
            else bundle_odd_scatter2<false, false, FORCE>(A, N, nb, ns, mas, mbs, act_a, act_b, h, pf);
        }
    }
    if constexpr (INLETS) {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets(p, ci, ia, ib)) {
            const NbrPair nb(p, ci.x, ci.y, ci.z, false);
            odd2_produce_bundle(p, nb, ci.n, ci.x, ci.y, ci.z, ia, ib);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// ============================== AA pattern, odd step, two cells =================================
// FLUID cells that are not special.  Population q goes to (q, x + c_q); on a solid link also to
// the own mirrored slot (opposite(q), x), which is the one the next even step reads.
// ma, mb: solid-link masks, zero for a cell that is not updated here.
template <int L, bool WALL, bool BOTH, bool FORCE, int Q = 0, typename S>
__device__ __forceinline__ void odd2_scatter(const Params& p, const NbrPair& nb, uint32_t n,
                                             uint32_t ma, uint32_t mb, bool act_a, bool act_b,
                                             const S& src, PairForce& pf) {
    Elem<L>* A = static_cast<Elem<L>*>(p.A);
    const uint32_t far = p.plane32[Q] + nb.template yz<Q, 1>(n);
    const float2 v = src.template get<Q>();
    if constexpr (WALL && Q > 0) {
        // each cell: neighbour slot, or its own mirrored slot on a solid link
        // every working cell writes its neighbour slot -- on a solid link that slot is the SOLID
        // cell's, read by nobody, and writing it keeps the sectors of the plane whole -- and on a
        // solid link also its own mirrored slot, the one the next even step reads
        const bool ba = solid_link<Q>(ma), bb = solid_link<Q>(mb);
        nb.template store<L, Q, 1, BOTH>(A + far, v, act_a, act_b);
        Elem<L>* own = A + (p.plane32[opp(Q)] + n);
        if (ba) st1s<L>(own, v.x);
        if (bb) st1s<L>(own + 1, v.y);
        if (FORCE) pf.template link<Q>(v, ba, bb);
    } else {
        nb.template store<L, Q, 1, BOTH>(A + far, v, act_a, act_b);
    }
    if constexpr (Q < 18) odd2_scatter<L, WALL, BOTH, FORCE, Q + 1>(p, nb, n, ma, mb, act_a, act_b, src, pf);
}

// AA odd step of INLET cells (producers): population q of the reservoir, f_eq,q(rho_in, u_in), to
// (q, s + c_q) -- where a FLUID cell's scatter leaves its population q for the neighbour's next
// even step -- for each INLET cell of the pair (ia, ib); a link leaving the domain through an OPEN
// face is dropped (its wrapped slot belongs to the boundary kernel's zero-gradient copies).
template <int L, int Q = 1>
__device__ __forceinline__ void odd2_produce(const Params& p, const NbrPair& nb, uint32_t n, int x,
                                             int y, int z, bool ia, bool ib) {
    Elem<L>* A = static_cast<Elem<L>*>(p.A);
    const uint32_t far = p.plane32[Q] + nb.template yz<Q, 1>(n);
    const bool yz_out = (cy(Q) != 0 && p.open[1] && y == (cy(Q) > 0 ? p.ny - 1 : 0)) ||
                        (cz(Q) != 0 && p.open[2] && z == (cz(Q) > 0 ? p.nz - 1 : 0));
    const bool xa_out = cx(Q) < 0 && p.open[0] && x == 0;
    const bool xb_out = cx(Q) > 0 && p.open[0] && x + 2 == p.nx;
    if (ia && !yz_out && !xa_out) st1<L>(A + (far + (uint32_t)nb.template xa<Q, 1>()), p.heq_in[Q]);
    if (ib && !yz_out && !xb_out) st1<L>(A + (far + (uint32_t)nb.template xb<Q, 1>()), p.heq_in[Q]);
    if constexpr (Q < 18) odd2_produce<L, Q + 1>(p, nb, n, x, y, z, ia, ib);
}

// WALLS = false: the grid has no solid link (its near-wall path compiled out, fewer registers and
// spills; the fp32 arrays and 4 blocks per SM stay: the packed half-precision form at 5 or 6 blocks
// spilled 60-160 bytes and was slower, fp16 periodic 512^3 odd step 2.26 / 2.55 ms against 2.02)
template <int L, bool WALLS>
constexpr int odd2_min_blocks() { return WALLS ? pair_min_blocks<L>(kPackedHalfOdd) : kOddBlocksNoWalls; }
template <int L, bool FORCE, bool BODY, bool INLETS, bool WALLS = true>
__global__ void __launch_bounds__(256, odd2_min_blocks<L, WALLS>()) k_aa_odd2(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const bool in = grid_pair(p, c);
    PairFlags f{0, 0, 0u, 0u};
    if (in) f = pair_flags(p, c.n, WALLS && p.any_solid_link != 0);
    const bool act_a = in && (f.fa & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
    const bool act_b = in && (f.fb & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
    if (!act_a) f.ma = 0u;
    if (!act_b) f.mb = 0u;
    // warp-uniform code paths: any solid link in the warp; every working thread owns two
    // working cells
    const bool wall = WALLS && __any_sync(0xffffffffu, (f.ma | f.mb) != 0u);
    const bool both = __all_sync(0xffffffffu, act_a == act_b);
    if ((act_a || act_b) && L == LAYOUT_STREAM_FP16 && kPackedHalfOdd) {
        // half-precision storage: the gathered pairs stay packed; each population is relaxed in
        // the scatter
        __half2 hh[19];
        {
            const NbrPair nb(p, c.x, c.y, c.z, false);
            if (wall) pair_gather_h<true, true>(p, nb, c.n, f.ma, f.mb, hh);
            else pair_gather_h<true, false>(p, nb, c.n, f.ma, f.mb, hh);
        }
        const Moments<Arith2> m = moments<Arith2, BODY>(HalfPairView{hh}, p);
        uint32_t ns = c.n, mas = f.ma, mbs = f.mb;
        int xs = c.x, ys = c.y, zs = c.z;
        asm volatile("" : "+r"(ns), "+r"(mas), "+r"(mbs), "+r"(xs), "+r"(ys), "+r"(zs)
                     : "f"(m.rho.x), "f"(m.rho.y));
        const NbrPair nb(p, xs, ys, zs, false);
        const RelaxSrc<BODY> src{m, hh, p};
        PairForce pf;
        if (wall) {
            if (both) odd2_scatter<L, true, true, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            else odd2_scatter<L, true, false, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            if (FORCE) pf.into(fx, fy, fz);
        } else {
            if (both) odd2_scatter<L, false, true, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            else odd2_scatter<L, false, false, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
        }
    } else if (act_a || act_b) {
        float2 h[19];
        {
            const NbrPair nb(p, c.x, c.y, c.z, false);
            if (wall) pair_gather<L, true, true>(p, nb, c.n, f.ma, f.mb, h);
            else pair_gather<L, true, false>(p, nb, c.n, f.ma, f.mb, h);
        }
        collide2<BODY>(h, p);
        // the scatter's geometry is formed after the collision (not held in registers across it)
        uint32_t ns = c.n, mas = f.ma, mbs = f.mb;
        int xs = c.x, ys = c.y, zs = c.z;
        asm volatile("" : "+r"(ns), "+r"(mas), "+r"(mbs), "+r"(xs), "+r"(ys), "+r"(zs)
                     : "f"(h[0].x), "f"(h[18].y));
        const NbrPair nb(p, xs, ys, zs, false);
        const ArraySrc src{h};
        PairForce pf;
        if (wall) {
            if (both) odd2_scatter<L, true, true, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            else odd2_scatter<L, true, false, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            if (FORCE) pf.into(fx, fy, fz);
        } else {
            if (both) odd2_scatter<L, false, true, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
            else odd2_scatter<L, false, false, FORCE>(p, nb, ns, mas, mbs, act_a, act_b, src, pf);
        }
    }
    if constexpr (INLETS) {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets(p, ci, ia, ib)) {
            const NbrPair nb(p, ci.x, ci.y, ci.z, false);
            odd2_produce<L>(p, nb, ci.n, ci.x, ci.y, ci.z, ia, ib);
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

// ============================== two buffers (A-B), two cells ====================================
// FROM_NATURAL: collide the natural state of every FLUID cell (B may equal A).  Otherwise pull-
// collide the FLUID cells that are not special.  Results go to (q, x) of B as aligned words, a
// special cell's slots included (its boundary kernel, launched after this one, overwrites them):
// every sector of B is then written whole.  Leaving those slots out, so that the boundary kernel
// could run at the same time, cost 8-13% on the sphere workload (partly written sectors filled
// from DRAM) for a 1-3% gain from the overlap.
// WALLS = false: the grid has no solid link (the near-wall gather and the momentum exchange
// compiled out; periodic 512^3 pull fp16 1.884 -> 1.847 ms, fp32 2.963 -> 2.945 ms; at 5 blocks
// per SM it spilled and was slower)
template <int L, bool FORCE, bool BODY, bool FROM_NATURAL, bool INLETS, bool WALLS = true>
__global__ void __launch_bounds__(256, 4) k_ab2(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const bool in = grid_pair<true>(p, c);
    PairFlags f{0, 0, 0u, 0u};
    if (in) f = pair_flags(p, c.n, WALLS && p.any_solid_link != 0 && (FORCE || !FROM_NATURAL));
    const uint8_t want = FROM_NATURAL ? TYPE_MASK : (TYPE_MASK | F_SPECIAL);
    const bool act_a = in && (f.fa & want) == T_FLUID;
    const bool act_b = in && (f.fb & want) == T_FLUID;
    const bool wall = WALLS && !FROM_NATURAL &&
                      __any_sync(0xffffffffu, (act_a || act_b) && (f.ma | f.mb) != 0u);
    Elem<L>* B = static_cast<Elem<L>*>(p.B);
    if (act_a || act_b) {
        float2 h[19];
        if (FROM_NATURAL) {
            const Elem<L>* A = static_cast<const Elem<L>*>(p.A);
#pragma unroll
            for (int q = 0; q < 19; ++q) h[q] = ld2<L>(A + (p.plane32[q] + c.n));
        } else {
            const NbrPair nb(p, c.x, c.y, c.z, true);
            if (wall) pair_gather<L, false, true>(p, nb, c.n, f.ma, f.mb, h);
            else pair_gather<L, false, false>(p, nb, c.n, f.ma, f.mb, h);
        }
        collide2<BODY>(h, p);
        uint32_t ns = c.n;
        asm volatile("" : "+r"(ns) : "f"(h[0].x), "f"(h[18].y));
#pragma unroll
        for (int q = 0; q < 19; ++q) st2<L>(B + (p.plane32[q] + ns), h[q]);
        if (FORCE) {
            if (WALLS && ((act_a && f.ma) || (act_b && f.mb))) {
                PairForce pf;
                pf.masks(act_a ? f.ma : 0u, act_b ? f.mb : 0u, h);
                pf.into(fx, fy, fz);
            }
            if (FROM_NATURAL && p.any_moving) {
                if (act_a && (f.fa & F_SPECIAL)) moving_forces(p, PairLane<0>{h}, c.x, c.y, c.z, fx, fy, fz);
                if (act_b && (f.fb & F_SPECIAL)) moving_forces(p, PairLane<1>{h}, c.x + 1, c.y, c.z, fx, fy, fz);
            }
        }
    } else if (in && p.B != p.A) {
        // no working cell: SOLID / MOVING_WALL slots are never read, special cells' are rewritten
        // by the boundary kernel and INLET cells' by the tail pass: zeros keep every sector of B
        // fully written
#pragma unroll
        for (int q = 0; q < 19; ++q) st2<L>(B + (p.plane32[q] + c.n), make_float2(0.f, 0.f));
    }
    if constexpr (INLETS) {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets<true>(p, ci, ia, ib)) pair_inlet_store<L, false>(p, p.B, ci.n, ia, ib);
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

// ============================== two buffers (A-B), bundle layout, two cells =====================
// The A-B steps in the bundle layout on an even nx.  The pull takes population q, member m of
// bundle (c_y, c_z), from the same member of the same bundle in the record of x - c_q: for a pair
// on one row the six elements lie in the records x - 1 .. x + 2, as 3 x + {-1, 1, 2, 3, 4, 6}
// relative to the row (one aligned word, 3 x + 2 .. 3 x + 3, and four elements).  The results go to
// the pair's own records, one aligned run of six elements per bundle of three (three words), as
// in the AA even step; the natural-state collision reads that run too.  Neighbour offsets clamp on
// OPEN axes (the zero-gradient source), as in the stream layout.  Measured against the one-cell
// pull with its stores staged through shared memory: 256^3 0.438 -> 0.385 ms, 128^3 0.061 ->
// 0.055 ms; 3 blocks per SM (80 registers) 1-2% ahead of 4 (64 registers, spilling).
template <bool WALL, int Q = 0>
__device__ __forceinline__ void bundle_pull_gather2(const float* A, uint32_t N, const NbrPair& nb,
                                                    uint32_t n, uint32_t ma, uint32_t mb,
                                                    float2 (&h)[19]) {
    if constexpr (bundle_j(Q) == 0) {
        // the source: this bundle on the row (y - c_y, z - c_z)
        const uint32_t r = nb.template yz<Q, -1>(n);
        if constexpr (bundle_size(Q) == 3) {
            constexpr int m0 = bundle_member(Q, 0), m1 = bundle_member(Q, 1), m2 = bundle_member(Q, 2);
            const uint32_t e = (uint32_t)bundle_off(Q) * N + 3u * r;
            if constexpr (WALL) {
                // on a solid link opposite(q) the cell's own slot (opposite(q), x) instead
                h[m0] = make_float2(A[bsel<m0>(ma, bidx<opp(m0)>(N, n), e + 3)],
                                    A[bsel<m0>(mb, bidx<opp(m0)>(N, n + 1), e + 3 * nb.wb)]);
                h[m1] = make_float2(A[bsel<m1>(ma, bidx<opp(m1)>(N, n), e + 1)],
                                    A[bsel<m1>(mb, bidx<opp(m1)>(N, n + 1), e + 4)]);
                h[m2] = make_float2(A[bsel<m2>(ma, bidx<opp(m2)>(N, n), e + 3 * nb.wa + 2)],
                                    A[bsel<m2>(mb, bidx<opp(m2)>(N, n + 1), e + 2)]);
            } else {
                const float2 w = ld2<LAYOUT_BUNDLE>(A + e + 2);  // (b's member 2, a's member 0)
                h[m0] = make_float2(w.y, A[e + 3 * nb.wb]);
                h[m1] = make_float2(A[e + 1], A[e + 4]);
                h[m2] = make_float2(A[e + 3 * nb.wa + 2], w.x);
            }
        } else {
            const uint32_t e = (uint32_t)bundle_off(Q) * N + r;
            if constexpr (WALL)
                h[Q] = make_float2(A[bsel<Q>(ma, bidx<opp(Q)>(N, n), e)],
                                   A[bsel<Q>(mb, bidx<opp(Q)>(N, n + 1), e + 1)]);
            else
                h[Q] = ld2<LAYOUT_BUNDLE>(A + e);
        }
    }
    if constexpr (Q < 18) bundle_pull_gather2<WALL, Q + 1>(A, N, nb, n, ma, mb, h);
}

// the pair's own records: [a0 a1 a2 b0 b1 b2] of a bundle of three as three words, one word for a
// bundle of one
template <int Q = 0>
__device__ __forceinline__ void bundle_store2(float* B, uint32_t N, uint32_t a, const float2 (&h)[19]) {
    if constexpr (bundle_j(Q) == 0) {
        float* e = B + ((uint32_t)bundle_off(Q) * N + a * (uint32_t)bundle_size(Q));
        if constexpr (bundle_size(Q) == 3) {
            const float2 v0 = h[bundle_member(Q, 0)], v1 = h[bundle_member(Q, 1)],
                         v2 = h[bundle_member(Q, 2)];
            st2<LAYOUT_BUNDLE>(e, make_float2(v0.x, v1.x));
            st2<LAYOUT_BUNDLE>(e + 2, make_float2(v2.x, v0.y));
            st2<LAYOUT_BUNDLE>(e + 4, make_float2(v1.y, v2.y));
        } else {
            st2<LAYOUT_BUNDLE>(e, h[Q]);
        }
    }
    if constexpr (Q < 18) bundle_store2<Q + 1>(B, N, a, h);
}

template <bool FORCE, bool BODY, bool FROM_NATURAL>
__global__ void __launch_bounds__(256, 3) k_ab2_bundle(Params p) {
    PairCoord c;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    const bool in = grid_pair<true>(p, c);
    PairFlags f{0, 0, 0u, 0u};
    if (in) f = pair_flags(p, c.n, p.any_solid_link != 0 && (FORCE || !FROM_NATURAL));
    const uint8_t want = FROM_NATURAL ? TYPE_MASK : (TYPE_MASK | F_SPECIAL);
    const bool act_a = in && (f.fa & want) == T_FLUID;
    const bool act_b = in && (f.fb & want) == T_FLUID;
    if (!act_a) f.ma = 0u;
    if (!act_b) f.mb = 0u;
    const bool wall = !FROM_NATURAL && __any_sync(0xffffffffu, (f.ma | f.mb) != 0u);
    float* B = static_cast<float*>(p.B);
    const uint32_t N = (uint32_t)p.N;
    if (act_a || act_b) {
        const float* A = static_cast<const float*>(p.A);
        float2 h[19];
        if (FROM_NATURAL) {
            bundle_gather2(A, N, c.n, h);
        } else {
            const NbrPair nb(p, c.x, c.y, c.z, true);
            if (wall) bundle_pull_gather2<true>(A, N, nb, c.n, f.ma, f.mb, h);
            else bundle_pull_gather2<false>(A, N, nb, c.n, f.ma, f.mb, h);
        }
        collide2<BODY>(h, p);
        uint32_t ns = c.n;
        asm volatile("" : "+r"(ns) : "f"(h[0].x), "f"(h[18].y));
        bundle_store2(B, N, ns, h);
        if (FORCE) {
            if (f.ma || f.mb) {
                PairForce pf;
                pf.masks(f.ma, f.mb, h);
                pf.into(fx, fy, fz);
            }
            if (FROM_NATURAL && p.any_moving) {
                if (act_a && (f.fa & F_SPECIAL)) moving_forces(p, PairLane<0>{h}, c.x, c.y, c.z, fx, fy, fz);
                if (act_b && (f.fb & F_SPECIAL)) moving_forces(p, PairLane<1>{h}, c.x + 1, c.y, c.z, fx, fy, fz);
            }
        }
    } else if (in && p.B != p.A) {
        // no working cell: SOLID / MOVING_WALL slots are never read, special cells' are rewritten
        // by the boundary kernel and INLET cells' by the tail pass: zeros keep every sector of B
        // fully written
        float2 z[19];
#pragma unroll
        for (int q = 0; q < 19; ++q) z[q] = make_float2(0.f, 0.f);
        bundle_store2(B, N, c.n, z);
    }
    {
        PairCoord ci;
        bool ia = false, ib = false;
        if (pair_inlets<true>(p, ci, ia, ib)) {
#pragma unroll
            for (int q = 0; q < 19; ++q) {
                if (ia) B[idx<LAYOUT_BUNDLE, uint32_t>(q, ci.n, N)] = p.heq_in[q];
                if (ib) B[idx<LAYOUT_BUNDLE, uint32_t>(q, ci.n + 1, N)] = p.heq_in[q];
            }
        }
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial, p.part_main);
}

}  // namespace lbm
