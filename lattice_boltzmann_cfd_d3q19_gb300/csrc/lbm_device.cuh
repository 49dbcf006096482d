// Device-side building blocks of the D3Q19 BGK step: velocity set, weights, layout addressing,
// per-link geometry and the collision.  Everything that depends on q is a constexpr function of
// q, so fully unrolled loops over the 19 populations fold it into immediates.
//
// Populations are stored SHIFTED: h_q = f_q - w_q (fp32).  At rest (rho = 1, u = 0) h = 0, and
// the values a step adds or subtracts are small against h, which keeps fp32 rounding of the
// near-unity density out of long runs.  The C ABI always exchanges absolute f.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace lbm {

// LAYOUT_STREAM_FP16: the stream layout with the shifted populations stored as IEEE half
// precision (arithmetic stays fp32); half the bytes per cell update.
enum : int { LAYOUT_STREAM = 0, LAYOUT_BUNDLE = 1, LAYOUT_COLLISION = 2, LAYOUT_STREAM_FP16 = 3 };
__host__ __device__ constexpr bool is_soa(int L) { return L == LAYOUT_STREAM || L == LAYOUT_STREAM_FP16; }
__host__ __device__ constexpr size_t elem_bytes(int L) { return L == LAYOUT_STREAM_FP16 ? 2 : 4; }

// internal flag byte: bits 0-1 cell type; for FLUID cells
//  bit 6 "special": a neighbour x + c_q is INLET or MOVING_WALL or lies beyond an OPEN face -- the
//        cell takes the general per-link path in the boundary kernels;
//  bit 7 "bulk": all 18 neighbours exist inside the domain (wrapped on periodic axes) and are
//        FLUID -- no link rule applies.
// FLUID cells that are neither have SOLID neighbours only; their links are described by the
// per-cell solid-link mask (bit q set when x + c_q, wrapped or clamped, is SOLID).
enum : uint8_t { T_FLUID = 0, T_SOLID = 1, T_INLET = 2, T_MOVING = 3, TYPE_MASK = 3,
                 F_SPECIAL = 0x40, F_BULK = 0x80 };

// what the population buffer holds between steps
enum : int {
    ST_NATURAL = 0,  // natural h_q(x) at slot (q, x)
    ST_POST_AA = 1,  // post-collision h*_q(x) at slot (opposite(q), x): AA after an even step
    ST_POST_AB = 2   // post-collision h*_q(x) at slot (q, x): two-buffer pull state
};

// ---- D3Q19 velocity set ---------------------------------------------------------------------
// Member order: rest, then each moving velocity followed by its opposite.  The velocity is coded
// as (cx+1) + 3 (cy+1) + 9 (cz+1).
__host__ __device__ constexpr int vcode(int q) {
    return q == 0 ? 13 : q == 1 ? 14 : q == 2 ? 12 : q == 3 ? 16 : q == 4 ? 10 : q == 5 ? 22
         : q == 6 ? 4 : q == 7 ? 17 : q == 8 ? 9 : q == 9 ? 23 : q == 10 ? 3 : q == 11 ? 25
         : q == 12 ? 1 : q == 13 ? 11 : q == 14 ? 15 : q == 15 ? 5 : q == 16 ? 21 : q == 17 ? 7
         : 19;
}
__host__ __device__ constexpr int cx(int q) { return vcode(q) % 3 - 1; }
__host__ __device__ constexpr int cy(int q) { return (vcode(q) / 3) % 3 - 1; }
__host__ __device__ constexpr int cz(int q) { return vcode(q) / 9 - 1; }
__host__ __device__ constexpr int opp(int q) { return q == 0 ? 0 : (q & 1) ? q + 1 : q - 1; }
// the same for a q known only at run time (one thread or lane per population)
__device__ __forceinline__ int c_rt(unsigned pos, unsigned neg, int q) {
    return (int)((pos >> q) & 1u) - (int)((neg >> q) & 1u);
}
__device__ __forceinline__ int cx_rt(int q) {
    return c_rt((1u << 1) | (1u << 7) | (1u << 9) | (1u << 13) | (1u << 15),
                (1u << 2) | (1u << 8) | (1u << 10) | (1u << 14) | (1u << 16), q);
}
__device__ __forceinline__ int cy_rt(int q) {
    return c_rt((1u << 3) | (1u << 7) | (1u << 11) | (1u << 14) | (1u << 17),
                (1u << 4) | (1u << 8) | (1u << 12) | (1u << 13) | (1u << 18), q);
}
__device__ __forceinline__ int cz_rt(int q) {
    return c_rt((1u << 5) | (1u << 9) | (1u << 11) | (1u << 16) | (1u << 18),
                (1u << 6) | (1u << 10) | (1u << 12) | (1u << 15) | (1u << 17), q);
}
__device__ __forceinline__ int opp_rt(int q) { return q == 0 ? 0 : (q & 1) ? q + 1 : q - 1; }
__host__ __device__ constexpr float wq(int q) {
    return q == 0 ? 1.0f / 3.0f : q <= 6 ? 1.0f / 18.0f : 1.0f / 36.0f;
}
__device__ __forceinline__ float wq_rt(int q) { return wq(q); }

// ---- layout addressing ------------------------------------------------------------------------
// STREAM (SoA): q*N + n.  COLLISION (AoS): n*19 + q.  BUNDLE (SoAoS): the populations sharing
// (cy, cz) form one bundle -- an x-row of the stencil, members ordered cx = -1, 0, +1 -- stored as
// boff*N + n*size + j.
__host__ __device__ constexpr int bundle_size(int q) { return (cy(q) == 0 || cz(q) == 0) ? 3 : 1; }
__host__ __device__ constexpr int bundle_off(int q) {
    return (cy(q) == 0 && cz(q) == 0) ? 0 : (cy(q) == 1 && cz(q) == 0) ? 3
         : (cy(q) == -1 && cz(q) == 0) ? 6 : (cy(q) == 0 && cz(q) == 1) ? 9
         : (cy(q) == 0 && cz(q) == -1) ? 12 : (cy(q) == 1 && cz(q) == 1) ? 15
         : (cy(q) == -1 && cz(q) == -1) ? 16 : (cy(q) == 1 && cz(q) == -1) ? 17 : 18;
}
__host__ __device__ constexpr int bundle_j(int q) { return bundle_size(q) == 3 ? cx(q) + 1 : 0; }

// Element offset of population q of cell n.
template <int L, typename I = size_t>
__host__ __device__ __forceinline__ I idx(int q, uint32_t n, I N) {
    if (is_soa(L)) return (I)q * N + (I)n;
    if (L == LAYOUT_COLLISION) return (I)n * (I)19 + (I)q;
    return (I)bundle_off(q) * N + (I)n * (I)bundle_size(q) + (I)bundle_j(q);
}
// In every layout population q of cell n sits at plane(q) + n * cell_stride(q), with
// plane(q) = idx(q, 0); opposite populations share their stride.
template <int L>
__host__ __device__ constexpr int cell_stride(int q) {
    return is_soa(L) ? 1 : L == LAYOUT_COLLISION ? 19 : bundle_size(q);
}

// Population storage access: element `off` of a buffer of layout L, as fp32.
template <int L, typename Off>
__device__ __forceinline__ float ld(const void* base, Off off) {
    if constexpr (L == LAYOUT_STREAM_FP16) return __half2float(static_cast<const __half*>(base)[off]);
    else return static_cast<const float*>(base)[off];
}
template <int L, typename Off>
__device__ __forceinline__ void st(void* base, Off off, float v) {
    if constexpr (L == LAYOUT_STREAM_FP16) static_cast<__half*>(base)[off] = __float2half_rn(v);
    else static_cast<float*>(base)[off] = v;
}
// runtime-q variant (off the hot path)
template <int L>
__host__ __device__ __forceinline__ size_t idx_rt(int q, uint32_t n, size_t N) {
    if (is_soa(L)) return (size_t)q * N + n;
    if (L == LAYOUT_COLLISION) return (size_t)n * 19u + (size_t)q;
    int s = 0, o = 0, j = 0;
    switch (q) {
#define LBM_BCASE(Q) case Q: s = bundle_size(Q); o = bundle_off(Q); j = bundle_j(Q); break;
        LBM_BCASE(0) LBM_BCASE(1) LBM_BCASE(2) LBM_BCASE(3) LBM_BCASE(4) LBM_BCASE(5)
        LBM_BCASE(6) LBM_BCASE(7) LBM_BCASE(8) LBM_BCASE(9) LBM_BCASE(10) LBM_BCASE(11)
        LBM_BCASE(12) LBM_BCASE(13) LBM_BCASE(14) LBM_BCASE(15) LBM_BCASE(16) LBM_BCASE(17)
        LBM_BCASE(18)
#undef LBM_BCASE
    }
    return (size_t)o * N + (size_t)n * (size_t)s + (size_t)j;
}

// ---- kernel parameters (passed by value) ---------------------------------------------------------
struct Params {
    void* A;               // buffer read (AA: the only buffer; A-B: source)
    void* B;               // A-B destination (may equal A for the in-place collision)
    const uint8_t* flags;  // internal flag bytes
    const uint32_t* mask;  // per-cell solid-link mask (0 for bulk cells)
    int any_solid_link;    // some FLUID cell has a SOLID neighbour (else every mask is 0)
    int any_moving;        // some FLUID cell has a MOVING_WALL neighbour
    int any_inlet;         // some cell is INLET (the step kernels run INLET cells as producers)
    int open_special;      // a link across an OPEN face makes a cell special (AA); the A-B pulls
                           // clamp such links in their main kernels instead
    int ghost_z;           // planes z = 0 and z = nz - 1 are ghost copies of neighbouring slabs
    const uint32_t* special;  // indices of the special FLUID cells
    uint32_t n_special;
    float* scratch;        // open-face pre-gathered values (AA odd step)
    double* partial;       // per-block momentum-exchange partial sums, 3 per block
    int* fault;            // set by a kernel whose bounded wait ran out (read by the host)
    uint32_t extra_tx;     // test hook: bytes a staged tile announces beyond its copies (normally 0)
    size_t part_main;      // first partial slot (triple) of an A-B step kernel's warps
    size_t part_special;   // first partial slot (triple) of the boundary kernels' warps
    int nx, ny, nz;
    int zrev;              // step kernels walk the z planes from nz - 1 down (alternated per step)
    // plane of an A-B step kernel's block (k_ab, k_ab2, k_ab_pull_staged, k_own_staged):
    // z = zbase + zstep * blockIdx.z, the same sweep as zrev for a launch over all planes, other
    // values for a launch over some planes (a slab's boundary or interior planes)
    int zbase, zstep;
    int open[3];           // axis has OPEN faces
    size_t N;
    size_t face_base[3][2];  // scratch offset of face (axis, side); 19 * area values each
    float omega;
    float g[3];
    float tau_g[3];        // tau g: equilibrium velocity shift of the Guo forcing
    float wk[19];          // -omega (tau - 1/2)^2 w_q (4.5 (c_q.g)^2 - 1.5 g.g)
    float heq_in[19];      // shifted inlet state f_eq(rho_in, u_in) - w
    float uw[3];           // velocity of the MOVING_WALL cells
    float wterm[19];       // 6 w_q (c_q . u_w): the moving-wall term of a population q leaving the wall
    // hot-path addressing: population q of cell n is pa[q][n * cell_stride(q)] in A and
    // pb[q][n * cell_stride(q)] in B; pdiff[q] = pa[q] - pa[opposite(q)] in elements
    void* pa[19];
    void* pb[19];
    long long pdiff[19];
    // compact addressing while every element offset fits in 32 bits (19 N <= 2^32): population q
    // of cell n is A[plane32[q] + n * cell_stride(q)] (one base, one 32-bit offset per access)
    uint32_t plane32[19];
};

// ---- collision -------------------------------------------------------------------------------------
// BGK with the second-order equilibrium (c_s^2 = 1/3) on shifted populations, plus Guo forcing
// when BODY: u = j/rho + g/2, F = rho g, source (1 - omega/2) w [3 (c - u).F + 9 (c.u)(c.F)].
// h[] holds h_q on entry and h*_q on exit.
//
// One cell (V = float) or two cells at once (V = float2, packed fp32x2 arithmetic: one
// instruction updates both cells).  Every operation is an explicit round-to-nearest add, multiply
// or fused multiply-add in a fixed order, so the two-cell form gives bit for bit the results of
// the one-cell form.
struct Arith1 {
    using V = float;
    static __device__ __forceinline__ V splat(float s) { return s; }
    static __device__ __forceinline__ V add(V a, V b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ V sub(V a, V b) { return __fsub_rn(a, b); }
    static __device__ __forceinline__ V mul(V a, V b) { return __fmul_rn(a, b); }
    static __device__ __forceinline__ V fma(V a, V b, V c) { return __fmaf_rn(a, b, c); }
    static __device__ __forceinline__ V neg(V a) { return -a; }
    // correctly rounded reciprocal, kept an opaque value: the compiler may otherwise evaluate a
    // product by it as a quotient
    static __device__ __forceinline__ V recip(V a) {
        float r = __frcp_rn(a);
        asm("" : "+f"(r));
        return r;
    }
};
// Packed fp32x2 operations written as PTX with an explicit .rn rounding: like the scalar
// __fadd_rn / __fmul_rn they are never contracted into a fused multiply-add.
struct Arith2 {
    using V = float2;
    static __device__ __forceinline__ unsigned long long pk(V a) {
        unsigned long long r;
        asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
        return r;
    }
    static __device__ __forceinline__ V up(unsigned long long r) {
        V a;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
        return a;
    }
    static __device__ __forceinline__ V splat(float s) { return make_float2(s, s); }
    static __device__ __forceinline__ V add(V a, V b) {
        unsigned long long d;
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
        return up(d);
    }
    static __device__ __forceinline__ V sub(V a, V b) {
        unsigned long long d;
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
        return up(d);
    }
    static __device__ __forceinline__ V mul(V a, V b) {
        unsigned long long d;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
        return up(d);
    }
    static __device__ __forceinline__ V fma(V a, V b, V c) {
        unsigned long long d;
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
        return up(d);
    }
    static __device__ __forceinline__ V neg(V a) { return make_float2(-a.x, -a.y); }
    static __device__ __forceinline__ V recip(V a) {
        float rx = __frcp_rn(a.x), ry = __frcp_rn(a.y);
        asm("" : "+f"(rx), "+f"(ry));
        return make_float2(rx, ry);
    }
};

// Population source of the collision: a one- or two-cell array, or two cells' stored half-precision
// values converted to fp32 where they are used (fewer registers held than an fp32 array).
template <typename V>
struct ArrayView {
    const V (&a)[19];
    __device__ __forceinline__ V operator()(int q) const { return a[q]; }
};
struct HalfPairView {
    const __half2 (&a)[19];
    __device__ __forceinline__ float2 operator()(int q) const { return __half22float2(a[q]); }
};

// sum over the populations whose velocity component along `axis` is `sign`, in q order
template <typename A, int axis, int sign, int Q = 1, bool FIRST = true, typename H>
__device__ __forceinline__ typename A::V side_sum(const H& h, typename A::V acc) {
    if constexpr (Q > 18) {
        return acc;
    } else {
        constexpr int c = axis == 0 ? cx(Q) : axis == 1 ? cy(Q) : cz(Q);
        if constexpr (c == sign) {
            typename A::V next;
            if constexpr (FIRST) next = h(Q);
            else next = A::add(acc, h(Q));
            return side_sum<A, axis, sign, Q + 1, false>(h, next);
        } else {
            return side_sum<A, axis, sign, Q + 1, FIRST>(h, acc);
        }
    }
}
template <typename A, int axis, typename H>
__device__ __forceinline__ typename A::V momentum(const H& h) {
    return A::sub(side_sum<A, axis, 1>(h, A::splat(0.f)), side_sum<A, axis, -1>(h, A::splat(0.f)));
}

// What the relaxation of every population needs from the cell's moments.
template <typename A>
struct Moments {
    typename A::V drho, rho, ux, uy, uz, nux, nuy, nuz, nuu15, nom;
};

template <typename A, bool BODY, typename H>
__device__ __forceinline__ Moments<A> moments(const H& h, const Params& p) {
    using V = typename A::V;
    Moments<A> m;
    V drho = h(0);
#pragma unroll
    for (int q = 1; q < 19; ++q) drho = A::add(drho, h(q));
    const V jx = momentum<A, 0>(h), jy = momentum<A, 1>(h), jz = momentum<A, 2>(h);
    m.drho = drho;
    m.rho = A::add(A::splat(1.0f), drho);
    const V inv = A::recip(m.rho);
    // Guo forcing, F = rho g, u = j/rho + g/2, source S_q = (1 - omega/2) d f_eq,q/du . g.
    // Because f_eq is quadratic in u, omega f_eq(u) + (1 - omega/2) d f_eq/du . g equals
    // omega f_eq(u + a g) - omega a^2 w rho (4.5 (c.g)^2 - 1.5 g.g) with a = tau - 1/2 exactly:
    // relax toward the equilibrium at j/rho + tau g and add rho wk_q, wk_q = -omega a^2 w_q
    // (4.5 (c_q.g)^2 - 1.5 g.g) (launch constants).
    if (BODY) {
        m.ux = A::fma(jx, inv, A::splat(p.tau_g[0]));
        m.uy = A::fma(jy, inv, A::splat(p.tau_g[1]));
        m.uz = A::fma(jz, inv, A::splat(p.tau_g[2]));
    } else {
        m.ux = A::mul(jx, inv);
        m.uy = A::mul(jy, inv);
        m.uz = A::mul(jz, inv);
    }
    m.nuu15 = A::mul(A::splat(-1.5f), A::fma(m.ux, m.ux, A::fma(m.uy, m.uy, A::mul(m.uz, m.uz))));
    m.nux = A::neg(m.ux);
    m.nuy = A::neg(m.uy);
    m.nuz = A::neg(m.uz);
    m.nom = A::splat(-p.omega);
    return m;
}

// Post-collision value of population q (a constant after unrolling) with pre-collision value h.
template <typename A, bool BODY>
__device__ __forceinline__ typename A::V relax_q(const Moments<A>& m, int q, typename A::V h,
                                                 const Params& p) {
    using V = typename A::V;
    // c_q . u: the signed velocity components, summed x, y, z
    V cu = A::splat(0.f);
    bool have = false;
    if (cx(q) != 0) { cu = cx(q) > 0 ? m.ux : m.nux; have = true; }
    if (cy(q) != 0) { const V t = cy(q) > 0 ? m.uy : m.nuy; cu = have ? A::add(cu, t) : t; have = true; }
    if (cz(q) != 0) { const V t = cz(q) > 0 ? m.uz : m.nuz; cu = have ? A::add(cu, t) : t; }
    // f_eq - w = w (rho - 1 + rho (3 cu + 4.5 cu^2 - 1.5 u.u))
    const V poly = q == 0 ? m.nuu15 : A::fma(cu, A::fma(A::splat(4.5f), cu, A::splat(3.0f)), m.nuu15);
    // h - (f_eq - w), then the relaxation h + (-omega) (h - h_eq)
    const V d = A::fma(A::splat(-wq(q)), A::fma(m.rho, poly, m.drho), h);
    V hn = A::fma(m.nom, d, h);
    if (BODY) hn = A::fma(m.rho, A::splat(p.wk[q]), hn);
    return hn;
}

template <typename A, bool BODY>
__device__ __forceinline__ void collide_t(typename A::V (&h)[19], const Params& p) {
    const Moments<A> m = moments<A, BODY>(ArrayView<typename A::V>{h}, p);
#pragma unroll
    for (int q = 0; q < 19; ++q) h[q] = relax_q<A, BODY>(m, q, h[q], p);
}

template <bool BODY>
__device__ __forceinline__ void collide(float (&h)[19], const Params& p) {
    collide_t<Arith1, BODY>(h, p);
}
template <bool BODY>
__device__ __forceinline__ void collide2(float2 (&h)[19], const Params& p) {
    collide_t<Arith2, BODY>(h, p);
}

// ---- momentum-exchange warp reduction ----------------------------------------------------------------
// Every thread of the warp must call this (full-warp shuffles, no block barrier, so a warp that
// is done leaves at once).  Lane 0 stores the warp's sum as one fp64 triple at slot
// slot_base + (linear block index) * (warps per block) + (warp in block).
constexpr int kWarpsPerBlock = 8;  // step kernels launch 256-thread blocks
// tiles of the collision layout's staged A-B pull: kTileX cells along x (a warp) by kTileY rows
constexpr int kTileX = 32;
constexpr int kTileY = 8;
__device__ __forceinline__ void warp_force(float fx, float fy, float fz, double* partial,
                                           size_t slot_base = 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        fx += __shfl_xor_sync(0xffffffffu, fx, o);
        fy += __shfl_xor_sync(0xffffffffu, fy, o);
        fz += __shfl_xor_sync(0xffffffffu, fz, o);
    }
    const int t = threadIdx.x + blockDim.x * threadIdx.y;
    if ((t & 31) == 0) {
        const size_t b = blockIdx.x + (size_t)gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z);
        const size_t w = slot_base + b * kWarpsPerBlock + (size_t)(t >> 5);
        partial[3 * w + 0] = (double)fx;
        partial[3 * w + 1] = (double)fy;
        partial[3 * w + 2] = (double)fz;
    }
}

// ---- momentum-exchange block reduction ----------------------------------------------------------------
// Every thread of the block must call this.  Warp shuffles, then one fp64 partial per block.
__device__ __forceinline__ void block_force(float fx, float fy, float fz, double* partial,
                                            size_t slot_base = 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        fx += __shfl_xor_sync(0xffffffffu, fx, o);
        fy += __shfl_xor_sync(0xffffffffu, fy, o);
        fz += __shfl_xor_sync(0xffffffffu, fz, o);
    }
    __shared__ float warp_sum[3][32];
    const int t = threadIdx.x + blockDim.x * threadIdx.y;
    const int nwarps = (blockDim.x * blockDim.y + 31) >> 5;
    if ((t & 31) == 0) {
        warp_sum[0][t >> 5] = fx;
        warp_sum[1][t >> 5] = fy;
        warp_sum[2][t >> 5] = fz;
    }
    __syncthreads();
    if (t == 0) {
        double s[3] = {0.0, 0.0, 0.0};
        for (int w = 0; w < nwarps; ++w)
            for (int a = 0; a < 3; ++a) s[a] += (double)warp_sum[a][w];
        const size_t b = slot_base + blockIdx.x +
                         (size_t)gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z);
        partial[3 * b + 0] = s[0];
        partial[3 * b + 1] = s[1];
        partial[3 * b + 2] = s[2];
    }
}

}  // namespace lbm
