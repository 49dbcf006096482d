// Instantiates the kernels for one population layout (LBM_LAYOUT) and fills its LayoutOps.
#pragma once

#include <algorithm>

#include "lbm_kernels.cuh"
#include "lbm_kernels_pair.cuh"
#include "lbm_kernels_tma.cuh"
#include "lbm_kernels_tile.cuh"
#include "lbm_kernels_boundary.cuh"
#include "lbm_launch.h"

namespace lbm {
namespace {

constexpr int L = LBM_LAYOUT;

template <bool F, bool B, typename I>
void launch_main(int kind, const Params& p, dim3 grid, dim3 block, cudaStream_t s) {
    switch (kind) {
        case K_AA_EVEN: k_aa_even<L, F, B, I><<<grid, block, 0, s>>>(p); break;
        case K_AA_ODD: k_aa_odd<L, F, B, I><<<grid, block, 0, s>>>(p); break;
        case K_AB_PULL: k_ab<L, F, B, false, I><<<grid, block, 0, s>>>(p); break;
        case K_AB_COLLIDE: k_ab<L, F, B, true, I><<<grid, block, 0, s>>>(p); break;
    }
}

// Addressing of the one-cell kernels: the neighbour-addressing kernels (AA odd, A-B) take one
// base pointer with 32-bit element offsets whenever all 19 N fit (fewer instructions per access);
// the even kernel, which already streams at the copy bandwidth, and larger grids use per-population
// plane pointers with 64-bit offsets.
template <bool F, bool B>
void launch_main_offsets(int kind, const Params& p, dim3 grid, dim3 block, cudaStream_t s) {
    // the steps that touch only a cell's own populations stage the collision layout's records
    // through shared memory (coalesced runs instead of elements 76 bytes apart)
    if constexpr (L == LAYOUT_COLLISION) {
        if (kind == K_AA_EVEN) {
            k_own_staged<F, B, true><<<grid, block, 0, s>>>(p);
            return;
        }
        if (kind == K_AB_COLLIDE) {
            k_own_staged<F, B, false><<<grid, block, 0, s>>>(p);
            return;
        }
    }
    if constexpr (!is_soa(L)) {
        if (kind == K_AB_PULL) {
            if (19 * p.N <= (size_t(1) << 32)) k_ab_pull_staged<L, F, B, uint32_t><<<grid, block, 0, s>>>(p);
            else k_ab_pull_staged<L, F, B, long long><<<grid, block, 0, s>>>(p);
            return;
        }
    }
    const bool compact = 19 * p.N <= (size_t(1) << 32) && kind != K_AA_EVEN;
    if (compact) launch_main<F, B, uint32_t>(kind, p, grid, block, s);
    else launch_main<F, B, long long>(kind, p, grid, block, s);
}

cudaError_t cells(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                  cudaStream_t s) {
    switch (kind) {
        case K_AA_EVEN:
        case K_AA_ODD:
        case K_AB_PULL:
        case K_AB_COLLIDE:
            if (force) {
                if (body) launch_main_offsets<true, true>(kind, p, grid, block, s);
                else launch_main_offsets<true, false>(kind, p, grid, block, s);
            } else {
                if (body) launch_main_offsets<false, true>(kind, p, grid, block, s);
                else launch_main_offsets<false, false>(kind, p, grid, block, s);
            }
            break;
        case K_STREAM:
            if (19 * p.N <= (size_t(1) << 32)) k_stream<L, uint32_t><<<grid, block, 0, s>>>(p);
            else k_stream<L, long long><<<grid, block, 0, s>>>(p);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Two-cell kernels (stream layouts; the bundle layout's even step; the caller checks an even nx and
// 19 N <= 2^32).
template <int LL, bool F, bool B, bool I>
void launch_pair_i(int kind, const Params& p, dim3 grid, dim3 block, cudaStream_t s) {
    switch (kind) {
        case K_AA_EVEN: k_aa_even2<LL, F, B, I><<<grid, block, 0, s>>>(p); break;
        case K_AA_ODD:
            // a grid without solid links takes the form without the near-wall path (fewer
            // registers and spills: periodic 512^3 odd step, fp16 2.087 -> 2.024 ms, fp32 3.061 ->
            // 3.044 ms)
            if (!p.any_solid_link)
                k_aa_odd2<LL, F, B, I, false><<<grid, block, 0, s>>>(p);
            else
                k_aa_odd2<LL, F, B, I><<<grid, block, 0, s>>>(p);
            break;
        case K_AB_PULL:
            if (!p.any_solid_link)
                k_ab2<LL, F, B, false, I, false><<<grid, block, 0, s>>>(p);
            else
                k_ab2<LL, F, B, false, I><<<grid, block, 0, s>>>(p);
            break;
        case K_AB_COLLIDE: k_ab2<LL, F, B, true, I><<<grid, block, 0, s>>>(p); break;
    }
}
// The half-precision instantiations without the INLET tail pass run where the domain has no
// inlet (measured: its never-taken epilogue cost the issue-bound fp16 kernels 4-5% at 512^3; the
// fp32 kernels, bound by memory, keep one instantiation).
template <int LL, bool F, bool B>
void launch_pair(int kind, const Params& p, dim3 grid, dim3 block, cudaStream_t s) {
    if constexpr (LL == LAYOUT_STREAM_FP16) {
        if (!p.any_inlet) {
            launch_pair_i<LL, F, B, false>(kind, p, grid, block, s);
            return;
        }
    }
    launch_pair_i<LL, F, B, true>(kind, p, grid, block, s);
}

template <int LL>
cudaError_t cells2_impl(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                        cudaStream_t s) {
    if constexpr (LL == LAYOUT_BUNDLE) {
        // the bundle layout's AA and A-B steps (two cells per thread); AB2's streaming pass is
        // one-cell
        if (kind == K_AA_EVEN) {
            if (force) {
                if (body) k_aa_even2_bundle<true, true><<<grid, block, 0, s>>>(p);
                else k_aa_even2_bundle<true, false><<<grid, block, 0, s>>>(p);
            } else {
                if (body) k_aa_even2_bundle<false, true><<<grid, block, 0, s>>>(p);
                else k_aa_even2_bundle<false, false><<<grid, block, 0, s>>>(p);
            }
        } else if (kind == K_AA_ODD) {
            const bool w = p.any_solid_link != 0;  // without solid links: no near-wall path
            if (force) {
                if (body) w ? k_aa_odd2_bundle<true, true, true><<<grid, block, 0, s>>>(p)
                            : k_aa_odd2_bundle<true, true, true, false><<<grid, block, 0, s>>>(p);
                else w ? k_aa_odd2_bundle<true, false, true><<<grid, block, 0, s>>>(p)
                       : k_aa_odd2_bundle<true, false, true, false><<<grid, block, 0, s>>>(p);
            } else {
                if (body) w ? k_aa_odd2_bundle<false, true, true><<<grid, block, 0, s>>>(p)
                            : k_aa_odd2_bundle<false, true, true, false><<<grid, block, 0, s>>>(p);
                else w ? k_aa_odd2_bundle<false, false, true><<<grid, block, 0, s>>>(p)
                       : k_aa_odd2_bundle<false, false, true, false><<<grid, block, 0, s>>>(p);
            }
        } else if (kind == K_AB_PULL || kind == K_AB_COLLIDE) {
            const bool nat = kind == K_AB_COLLIDE;
            if (force) {
                if (body) nat ? k_ab2_bundle<true, true, true><<<grid, block, 0, s>>>(p)
                              : k_ab2_bundle<true, true, false><<<grid, block, 0, s>>>(p);
                else nat ? k_ab2_bundle<true, false, true><<<grid, block, 0, s>>>(p)
                         : k_ab2_bundle<true, false, false><<<grid, block, 0, s>>>(p);
            } else {
                if (body) nat ? k_ab2_bundle<false, true, true><<<grid, block, 0, s>>>(p)
                              : k_ab2_bundle<false, true, false><<<grid, block, 0, s>>>(p);
                else nat ? k_ab2_bundle<false, false, true><<<grid, block, 0, s>>>(p)
                         : k_ab2_bundle<false, false, false><<<grid, block, 0, s>>>(p);
            }
        } else {
            return cudaErrorNotSupported;
        }
        return cudaGetLastError();
    } else if constexpr (!is_soa(LL)) {
        return cudaErrorNotSupported;
    } else {
        if (kind != K_AA_EVEN && kind != K_AA_ODD && kind != K_AB_PULL && kind != K_AB_COLLIDE)
            return cudaErrorInvalidValue;
        if (force) {
            if (body) launch_pair<LL, true, true>(kind, p, grid, block, s);
            else launch_pair<LL, true, false>(kind, p, grid, block, s);
        } else {
            if (body) launch_pair<LL, false, true>(kind, p, grid, block, s);
            else launch_pair<LL, false, false>(kind, p, grid, block, s);
        }
        return cudaGetLastError();
    }
}

cudaError_t cells2(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                   cudaStream_t s) {
    return cells2_impl<L>(kind, p, force, body, grid, block, s);
}

// TMA-staged AA odd kernel (stream layouts; the caller checks 16 | nx <= 512 and 19 N <= 2^32).
// The dynamic shared-memory limit is raised once per device and instantiation.
template <int LL, bool F, bool B>
cudaError_t launch_tma(const Params& p, unsigned grid, cudaStream_t s) {
    constexpr int kMaxDevices = 64;
    static bool raised[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!raised[dev]) {
        e = cudaFuncSetAttribute(k_aa_odd_tma<LL, F, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)TmaStage<LL>::total);
        if (e != cudaSuccess) return e;
        raised[dev] = true;
    }
    k_aa_odd_tma<LL, F, B><<<grid, kTmaThreads, TmaStage<LL>::total, s>>>(p);
    return cudaGetLastError();
}

template <int LL>
cudaError_t odd_tma_impl(const Params& p, bool force, bool body, unsigned grid, cudaStream_t s) {
    if constexpr (!is_soa(LL)) {
        return cudaErrorNotSupported;
    } else {
        if (force) return body ? launch_tma<LL, true, true>(p, grid, s) : launch_tma<LL, true, false>(p, grid, s);
        return body ? launch_tma<LL, false, true>(p, grid, s) : launch_tma<LL, false, false>(p, grid, s);
    }
}

cudaError_t odd_tma(const Params& p, bool force, bool body, unsigned grid, cudaStream_t s) {
    return odd_tma_impl<L>(p, force, body, grid, s);
}

// 2.5D-tiled A-B pull of the collision layout (the caller checks 32 | nx and 19 N <= 2^32)
template <int LL>
cudaError_t ab_pull_tile_impl(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s) {
    if constexpr (LL != LAYOUT_COLLISION) {
        return cudaErrorNotSupported;
    } else {
        const bool w = p.any_solid_link != 0;  // without solid links: no bounce-back selects
        if (force) {
            if (body) w ? k_ab_pull_tile<true, true><<<grid, kTileThreads, kTileSmemBytes, s>>>(p)
                        : k_ab_pull_tile<true, true, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p);
            else w ? k_ab_pull_tile<true, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p)
                   : k_ab_pull_tile<true, false, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p);
        } else {
            if (body) w ? k_ab_pull_tile<false, true><<<grid, kTileThreads, kTileSmemBytes, s>>>(p)
                        : k_ab_pull_tile<false, true, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p);
            else w ? k_ab_pull_tile<false, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p)
                   : k_ab_pull_tile<false, false, false><<<grid, kTileThreads, kTileSmemBytes, s>>>(p);
        }
        return cudaGetLastError();
    }
}
cudaError_t ab_pull_tile(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s) {
    return ab_pull_tile_impl<L>(p, force, body, grid, s);
}
template <int LL>
cudaError_t aa_odd_tile_impl(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s) {
    if constexpr (LL != LAYOUT_COLLISION) {
        return cudaErrorNotSupported;
    } else {
        const bool w = p.any_solid_link != 0;
        if (force) {
            if (body) w ? k_aa_odd_tile<true, true><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p)
                        : k_aa_odd_tile<true, true, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p);
            else w ? k_aa_odd_tile<true, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p)
                   : k_aa_odd_tile<true, false, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p);
        } else {
            if (body) w ? k_aa_odd_tile<false, true><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p)
                        : k_aa_odd_tile<false, true, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p);
            else w ? k_aa_odd_tile<false, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p)
                   : k_aa_odd_tile<false, false, false><<<grid, kTileThreads, kOddTileSmemBytes, s>>>(p);
        }
        return cudaGetLastError();
    }
}
cudaError_t aa_odd_tile(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s) {
    return aa_odd_tile_impl<L>(p, force, body, grid, s);
}
template <int LL>
cudaError_t tile_prepare_impl() {
    if constexpr (LL != LAYOUT_COLLISION) {
        return cudaSuccess;
    } else {
        const int bytes = (int)kTileSmemBytes;
        cudaError_t e = cudaFuncSetAttribute(k_ab_pull_tile<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<true, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_ab_pull_tile<false, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        const int odd = (int)kOddTileSmemBytes;
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<true, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<false, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_aa_odd_tile<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, odd);
        return e;
    }
}
cudaError_t tile_prepare() { return tile_prepare_impl<L>(); }

unsigned blocks_for(size_t count) { return (unsigned)((count + 255) / 256); }

#define LBM_LAUNCH_SPECIAL(KERNEL)                                                     \
    do {                                                                               \
        if (force) {                                                                   \
            if (body) KERNEL<L, true, true><<<grid, 256, 0, s>>>(p);                   \
            else KERNEL<L, true, false><<<grid, 256, 0, s>>>(p);                       \
        } else {                                                                       \
            if (body) KERNEL<L, false, true><<<grid, 256, 0, s>>>(p);                  \
            else KERNEL<L, false, false><<<grid, 256, 0, s>>>(p);                      \
        }                                                                              \
    } while (0)

cudaError_t special(int kind, const Params& p, bool force, bool body, cudaStream_t s) {
    if (p.n_special == 0) return cudaSuccess;
    // one warp per special cell (8 per block) for the collision kernels
    const unsigned grid = (p.n_special + kSpecialCellsPerBlock - 1) / kSpecialCellsPerBlock;
    switch (kind) {
        case K_AA_ODD: LBM_LAUNCH_SPECIAL(k_aa_odd_special); break;
        case K_AB_PULL: LBM_LAUNCH_SPECIAL(k_ab_special); break;
        case K_STREAM: k_stream_special<L><<<blocks_for(p.n_special), 256, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
#undef LBM_LAUNCH_SPECIAL

cudaError_t pregather(const Params& p, cudaStream_t s) {
    size_t area = 0;
    if (p.open[0]) area = std::max(area, (size_t)p.ny * p.nz);
    if (p.open[1]) area = std::max(area, (size_t)p.nx * p.nz);
    if (p.open[2]) area = std::max(area, (size_t)p.nx * p.ny);
    if (area == 0) return cudaSuccess;
    k_pregather<L><<<dim3(blocks_for(5 * area), 6), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t pack(const Params& p, const float* in, size_t i0, size_t count, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    k_pack<L><<<blocks_for(count), 256, 0, s>>>(p, in, i0, count);
    return cudaGetLastError();
}

cudaError_t unpack(const Params& p, int state, float* out, size_t i0, size_t count,
                   cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    k_unpack<L><<<blocks_for(count), 256, 0, s>>>(p, state, out, i0, count);
    return cudaGetLastError();
}

cudaError_t equilibrium(const Params& p, const float* rho, const float* u0, const float* u1,
                        const float* u2, uint32_t n0, uint32_t count, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    k_equilibrium<L><<<blocks_for(count), 256, 0, s>>>(p, rho, u0, u1, u2, n0, count);
    return cudaGetLastError();
}

cudaError_t macro(const Params& p, int state, const float inlet[4], float* rho, float* u0,
                  float* u1, float* u2, uint32_t n0, uint32_t count, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    k_macro<L><<<blocks_for(count), 256, 0, s>>>(p, state, inlet[0], inlet[1], inlet[2],
                                                   inlet[3], rho, u0, u1, u2, n0, count);
    return cudaGetLastError();
}

cudaError_t check_finite(const Params& p, int* bad, dim3 grid, dim3 block, cudaStream_t s) {
    k_check_finite<L><<<grid, block, 0, s>>>(p, bad);
    return cudaGetLastError();
}

cudaError_t fill_inlet(const Params& p, int state, dim3 grid, dim3 block, cudaStream_t s) {
    k_fill_inlet<L><<<grid, block, 0, s>>>(p, state);
    return cudaGetLastError();
}

cudaError_t halo_pack(const Params& p, void* lo, void* hi, cudaStream_t s) {
    k_halo_pack<L><<<blocks_for(10 * (size_t)p.nx * p.ny), 256, 0, s>>>(
        p, 1, p.nz - 2, static_cast<Stored<L>*>(lo), static_cast<Stored<L>*>(hi));
    return cudaGetLastError();
}

cudaError_t halo_unpack(const Params& p, const void* below, const void* above, cudaStream_t s) {
    k_halo_unpack<L><<<blocks_for(10 * (size_t)p.nx * p.ny), 256, 0, s>>>(
        p, static_cast<const Stored<L>*>(below), static_cast<const Stored<L>*>(above));
    return cudaGetLastError();
}

const LayoutOps kOps = {cells, cells2, odd_tma, ab_pull_tile, aa_odd_tile, tile_prepare, special, pregather, pack, unpack,
                        equilibrium, macro, check_finite, fill_inlet, halo_pack, halo_unpack};

}  // namespace
}  // namespace lbm
