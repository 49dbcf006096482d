// AA odd step with the gather staged through shared memory by TMA bulk copies (stream layouts,
// 16 | nx <= 512, 19 N <= 2^32).
//
// Persistent CTAs (one per SM) walk tiles of whole x-rows, R = floor(512 / nx) rows per tile.
// Along a velocity with c_x != 0 the sources of a row's cells are the cells of ONE source row
// (y - c_y, z - c_z) shifted by -c_x with periodic wrap in x, so every population plane of a tile
// is staged as exact, 16-byte-aligned rows: per tile and per plane one bulk copy per source row,
// and -- when the domain has solid links -- one bulk copy of the tile's own rows (the mirrored
// slots a solid link reads instead), plus the tile's flag bytes and solid-link masks.  Two stages
// alternate: while the CTA computes one tile from shared memory, the copies of the next are in
// flight (an mbarrier per stage counts their bytes).  The collision and the scatter are those of
// the two-cell kernel (one thread, two x-adjacent cells; stores straight to global memory).
//
// No race: in the AA odd step a cell reads and writes exactly its own 19 slots ("GPU lattice
// Boltzmann: streaming layout and performance", "In place"), so a tile's slots are written only
// by that tile, after they were staged.  The own rows also hold slots of cells in other tiles that
// may be written meanwhile; those elements are never used (only a cell's own mirrored slots are).
//
// Every wait on a stage's mbarrier is bounded (kWaitNs of wall time): on a timeout the whole CTA
// records kFaultWait in *p.fault, waits (bounded again) for the copies it still has in flight,
// and returns; the host reports the flag at its next synchronising call.
#pragma once

#include "lbm_kernels_pair.cuh"

namespace lbm {

constexpr int kTmaCells = 512;      // cells per tile (R whole rows, R * nx <= 512)
constexpr int kTmaThreads = 256;    // one thread per cell pair
constexpr unsigned long long kWaitNs = 2000000000ull;  // a stage wait gives up after 2 s
constexpr int kFaultWait = 1;

// shared-memory stage: far rows [19][T], own rows [19][T] (solid links only), flag bytes [T],
// solid-link masks [T]; T = kTmaCells elements.  The mbarriers follow the two stages.
template <int L>
struct TmaStage {
    static constexpr size_t far_bytes = 19u * kTmaCells * sizeof(Elem<L>);
    static constexpr size_t own_off = far_bytes;
    static constexpr size_t flags_off = own_off + far_bytes;
    static constexpr size_t mask_off = flags_off + kTmaCells;
    static constexpr size_t bytes = mask_off + kTmaCells * 4u;
    static constexpr size_t total = 2 * bytes + 16;  // two stages + two mbarriers
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// true once the phase with parity `parity` of the barrier has completed
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// bounded wait; false when kWaitNs ran out
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}
// bulk copy global -> shared (16-byte aligned, size a multiple of 16), completing on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tile geometry: R rows of nx cells; tile t covers rows [t R, min(t R + R, ny nz)).
struct TmaTiles {
    int R, rows_total, tiles;
    __device__ __forceinline__ TmaTiles(const Params& p) {
        R = kTmaCells / p.nx;
        rows_total = p.ny * p.nz;
        tiles = (rows_total + R - 1) / R;
    }
};

// Thread 0: issue the copies of tile t into stage `st` (its mbarrier `bar`).  One thread issues
// every copy (a form that spread them over the lanes of a warp never saw all of its copies
// arrive).
template <int L>
__device__ __forceinline__ void tma_issue(const Params& p, const TmaTiles& tg, int t,
                                         unsigned char* st, uint64_t* bar) {
    using E = Elem<L>;
    const E* A = static_cast<const E*>(p.A);
    const int r0 = t * tg.R;
    const int rows = min(tg.R, tg.rows_total - r0);
    const uint32_t row_bytes = (uint32_t)p.nx * sizeof(E);
    const uint32_t cells = (uint32_t)rows * (uint32_t)p.nx;
    const bool links = p.any_solid_link != 0;
    uint32_t bytes = 19u * rows * row_bytes + cells;
    if (links) bytes += 18u * rows * row_bytes + 4u * cells;
    // the stage was last read by every thread (a barrier precedes this call); order those
    // generic-proxy reads before the async-proxy writes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, bytes + p.extra_tx);
    E* far = reinterpret_cast<E*>(st);
    E* own = reinterpret_cast<E*>(st + TmaStage<L>::own_off);
    const uint32_t n0 = (uint32_t)r0 * (uint32_t)p.nx;
#pragma unroll
    for (int q = 0; q < 19; ++q) {
        // population q of row (y, z) pulls from row (y - c_y, z - c_z) of plane opposite(q)
        const int po = opp(q);
        for (int rr = 0; rr < rows; ++rr) {
            const int r = r0 + rr;
            int y = r % p.ny - cy(q), z = r / p.ny - cz(q);
            y = y < 0 ? y + p.ny : y >= p.ny ? y - p.ny : y;
            z = z < 0 ? z + p.nz : z >= p.nz ? z - p.nz : z;
            const uint32_t src = p.plane32[po] + ((uint32_t)y + (uint32_t)p.ny * (uint32_t)z) * (uint32_t)p.nx;
            bulk_g2s(far + (size_t)q * kTmaCells + (size_t)rr * p.nx, A + src, row_bytes, bar);
        }
        if (links && q > 0)
            bulk_g2s(own + (size_t)q * kTmaCells, A + (p.plane32[q] + n0), rows * row_bytes, bar);
    }
    bulk_g2s(st + TmaStage<L>::flags_off, p.flags + n0, cells, bar);
    if (links) bulk_g2s(st + TmaStage<L>::mask_off, p.mask + n0, 4u * cells, bar);
}

// population q of the pair (x, x + 1) in tile row rr, from the staged rows
template <int L, int Q = 0>
__device__ __forceinline__ void tma_gather(const unsigned char* st, int j, int x, int nx,
                                           uint32_t ma, uint32_t mb, bool links, float2 (&h)[19]) {
    using E = Elem<L>;
    const E* row = reinterpret_cast<const E*>(st) + (size_t)Q * kTmaCells + (j - x);  // row start
    float2 v;
    constexpr int sx = -cx(Q);  // source x offset
    if constexpr (sx == 0) {
        v = ld2<L>(row + x);
    } else if constexpr (sx < 0) {
        v = make_float2(ld1<L>(row + (x == 0 ? nx - 1 : x - 1)), ld1<L>(row + x));
    } else {
        v = make_float2(ld1<L>(row + x + 1), ld1<L>(row + (x + 2 == nx ? 0 : x + 2)));
    }
    if constexpr (Q > 0) {
        if (links) {
            // a solid link reads the cell's own mirrored slot (q, x) instead
            const float2 o = ld2<L>(reinterpret_cast<const E*>(st + TmaStage<L>::own_off) +
                                    (size_t)Q * kTmaCells + j);
            if (solid_link<opp(Q)>(ma)) v.x = o.x;
            if (solid_link<opp(Q)>(mb)) v.y = o.y;
        }
    }
    h[Q] = v;
    if constexpr (Q < 18) tma_gather<L, Q + 1>(st, j, x, nx, ma, mb, links, h);
}

template <int L, bool FORCE, bool BODY>
__global__ void __launch_bounds__(kTmaThreads, 1) k_aa_odd_tma(Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage[2] = {smem, smem + TmaStage<L>::bytes};
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * TmaStage<L>::bytes);
    const TmaTiles tg(p);
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // prologue: the CTA's first two tiles.  pending[s]: stage s has copies in flight, whose
    // completion is the barrier phase with parity phase[s]
    bool pending[2] = {false, false};
    uint32_t phase[2] = {0u, 0u};
    for (int s = 0; s < 2; ++s) {
        const int t = blockIdx.x + s * gridDim.x;
        if (t < tg.tiles) {
            if (tid == 0) tma_issue<L>(p, tg, t, stage[s], &bar[s]);
            pending[s] = true;
        }
    }

    float fx = 0.f, fy = 0.f, fz = 0.f;
    bool fault = false;
    int k = 0;
    for (int t = blockIdx.x; t < tg.tiles; t += gridDim.x, ++k) {
        const int s = k & 1;
        const bool ok = mbar_wait(&bar[s], phase[s]);
        // the same decision in every thread of the CTA
        if (__syncthreads_or(!ok)) {
            fault = true;
            break;
        }
        pending[s] = false;
        phase[s] ^= 1u;
        const unsigned char* st = stage[s];
        const int r0 = t * tg.R;
        const int cells = min(tg.R, tg.rows_total - r0) * p.nx;
        const int j = 2 * tid;  // first cell of the pair within the tile
        const bool in = j < cells;
        const int x = j % p.nx;
        const int r = r0 + j / p.nx;
        const uint32_t n = (uint32_t)r * (uint32_t)p.nx + (uint32_t)x;
        uint8_t fa = 0, fb = 0;
        uint32_t ma = 0u, mb = 0u;
        if (in) {
            fa = st[TmaStage<L>::flags_off + j];
            fb = st[TmaStage<L>::flags_off + j + 1];
            if (p.any_solid_link) {
                const uint2 m = *reinterpret_cast<const uint2*>(st + TmaStage<L>::mask_off + 4 * j);
                ma = m.x;
                mb = m.y;
            }
        }
        const bool act_a = in && (fa & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
        const bool act_b = in && (fb & (TYPE_MASK | F_SPECIAL)) == T_FLUID;
        if (!act_a) ma = 0u;
        if (!act_b) mb = 0u;
        const bool wall = __any_sync(0xffffffffu, (ma | mb) != 0u);
        const bool both = __all_sync(0xffffffffu, act_a == act_b);
        if (act_a || act_b) {
            float2 h[19];
            tma_gather<L>(st, j, x, p.nx, ma, mb, p.any_solid_link != 0, h);
            collide2<BODY>(h, p);
            const NbrPair nb(p, x, r % p.ny, r / p.ny, false);
            const ArraySrc src{h};
            PairForce pf;
            if (wall) {
                if (both) odd2_scatter<L, true, true, FORCE>(p, nb, n, ma, mb, act_a, act_b, src, pf);
                else odd2_scatter<L, true, false, FORCE>(p, nb, n, ma, mb, act_a, act_b, src, pf);
                if (FORCE) pf.into(fx, fy, fz);
            } else {
                if (both) odd2_scatter<L, false, true, FORCE>(p, nb, n, ma, mb, act_a, act_b, src, pf);
                else odd2_scatter<L, false, false, FORCE>(p, nb, n, ma, mb, act_a, act_b, src, pf);
            }
        }
        // INLET cells of the tile: producers, as in the register kernel
        const bool inl_a = is_inlet(p, in, fa), inl_b = is_inlet(p, in, fb);
        if (inl_a || inl_b) {
            const NbrPair nb(p, x, r % p.ny, r / p.ny, false);
            odd2_produce<L>(p, nb, n, x, r % p.ny, r / p.ny, inl_a, inl_b);
        }
        // every thread is done with stage s before it is refilled
        __syncthreads();
        const int t2 = t + 2 * (int)gridDim.x;
        if (t2 < tg.tiles) {
            if (tid == 0) tma_issue<L>(p, tg, t2, stage[s], &bar[s]);
            pending[s] = true;
        }
    }
    if (fault) {
        if (tid == 0) atomicExch(p.fault, kFaultWait);
        // copies still in flight must land before the CTA's shared memory is released
        for (int s = 0; s < 2; ++s)
            if (pending[s]) mbar_wait(&bar[s], phase[s]);
        return;
    }
    if (FORCE) warp_force(fx, fy, fz, p.partial);
}

}  // namespace lbm
