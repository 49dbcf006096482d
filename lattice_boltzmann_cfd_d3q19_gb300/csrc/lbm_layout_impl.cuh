// Instantiates the kernels for one population layout (LBM_LAYOUT) and fills its LayoutOps.
#pragma once

#include "lbm_kernels.cuh"
#include "lbm_launch.h"

namespace lbm {
namespace {

constexpr int L = LBM_LAYOUT;

#define LBM_LAUNCH_FB(KERNEL, EXTRA)                                                   \
    do {                                                                               \
        if (force) {                                                                   \
            if (body) KERNEL<L, true, true EXTRA><<<grid, block, 0, s>>>(p);           \
            else KERNEL<L, true, false EXTRA><<<grid, block, 0, s>>>(p);               \
        } else {                                                                       \
            if (body) KERNEL<L, false, true EXTRA><<<grid, block, 0, s>>>(p);          \
            else KERNEL<L, false, false EXTRA><<<grid, block, 0, s>>>(p);              \
        }                                                                              \
    } while (0)
#define LBM_COMMA ,

cudaError_t cells(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                  cudaStream_t s) {
    switch (kind) {
        case K_AA_EVEN: LBM_LAUNCH_FB(k_aa_even, ); break;
        case K_AA_ODD: LBM_LAUNCH_FB(k_aa_odd, ); break;
        case K_AB_PULL: LBM_LAUNCH_FB(k_ab, LBM_COMMA false); break;
        case K_AB_COLLIDE: LBM_LAUNCH_FB(k_ab, LBM_COMMA true); break;
        case K_STREAM: k_stream<L><<<grid, block, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

unsigned blocks_for(size_t count) { return (unsigned)((count + 255) / 256); }

cudaError_t pregather(const Params& p, int axis, int side, cudaStream_t s) {
    const size_t area = axis == 0 ? (size_t)p.ny * p.nz
                      : axis == 1 ? (size_t)p.nx * p.nz : (size_t)p.nx * p.ny;
    k_pregather<L><<<blocks_for(19 * area), 256, 0, s>>>(p, axis, side);
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

const LayoutOps kOps = {cells, pregather, pack, unpack, equilibrium, macro, check_finite};

#undef LBM_LAUNCH_FB
#undef LBM_COMMA
}  // namespace
}  // namespace lbm
