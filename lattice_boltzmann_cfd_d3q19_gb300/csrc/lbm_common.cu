// Layout-independent kernels: flag validation and classification, force finalisation.
#include "lbm_kernels.cuh"
#include "lbm_launch.h"

namespace lbm {
namespace {

__global__ void __launch_bounds__(256) k_validate_types(const uint8_t* types, size_t N, int* bad) {
    const size_t n = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n < N && types[n] > T_MOVING) *bad = 1;
}

// Internal flags and solid-link masks.  For a FLUID cell: mask bit q when x + c_q (wrapped, or
// clamped at an OPEN face) is SOLID; F_SPECIAL when some x + c_q is MOVING_WALL or, in the AA
// scheme (p.open_special), lies beyond an OPEN face; F_BULK when no link rule applies at all.
// INLET neighbours need no special path: INLET cells are producers in the step kernels (their
// slots carry f_eq(rho_in, u_in) where a FLUID neighbour's post-collision values would be), and
// the A-B pulls clamp links across an OPEN face in their main kernels.
// count[0]: special cells; count[1]: FLUID cells with a SOLID link; count[2]: FLUID cells with a
// MOVING_WALL link; count[3]: INLET cells
__global__ void __launch_bounds__(256) k_classify(Params p, const uint8_t* types, uint8_t* flags,
                                                  uint32_t* mask, uint32_t* count) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= p.nx || y >= p.ny) return;
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    const uint8_t t = types[n];
    uint8_t out = t;
    uint32_t m = 0;
    if (t == T_INLET) atomicAdd(count + 3, 1u);
    // a ghost plane's cells are stepped like the others, but their results are replaced by the
    // neighbouring slab's and they take no part in the momentum exchange: no links, never special
    const bool ghost = p.ghost_z && (z == 0 || z == p.nz - 1);
    if (t == T_FLUID && !ghost) {
        bool special = false, moving = false, plain = true;
        for (int q = 1; q < 19; ++q) {
            const Link s = link_cell(p, x, y, z, cx(q), cy(q), cz(q));
            const uint8_t ts = types[s.cell];
            if ((s.face >= 0 && p.open_special) || ts == T_MOVING) special = true;
            if (s.face >= 0 || ts != T_FLUID) plain = false;
            if (ts == T_MOVING) moving = true;
            if (ts == T_SOLID) m |= 1u << q;
        }
        if (moving) atomicAdd(count + 2, 1u);
        if (special) {
            out |= F_SPECIAL;
            atomicAdd(count, 1u);
        } else if (plain) {
            out |= F_BULK;
        }
        if (m != 0) atomicAdd(count + 1, 1u);
    }
    flags[n] = out;
    mask[n] = m;
}

__global__ void __launch_bounds__(256) k_list_special(Params p, const uint8_t* flags,
                                                      uint32_t* list, uint32_t* count) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= p.nx || y >= p.ny) return;
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    if (flags[n] & F_SPECIAL) list[atomicAdd(count, 1u)] = n;
}

// Stage 1: block b sums the partials of chunk b in a fixed order (thread-strided, then a tree).
// Stage 2: one block sums the stage values the same way.
__global__ void __launch_bounds__(256) k_force_sum(const double* partial, size_t nblocks,
                                                   size_t chunk, double* out) {
    __shared__ double s[3][256];
    const int t = threadIdx.x;
    const size_t b0 = (size_t)blockIdx.x * chunk;
    const size_t b1 = b0 + chunk < nblocks ? b0 + chunk : nblocks;
    double a0 = 0.0, a1 = 0.0, a2 = 0.0;
    for (size_t b = b0 + t; b < b1; b += 256) {
        a0 += partial[3 * b + 0];
        a1 += partial[3 * b + 1];
        a2 += partial[3 * b + 2];
    }
    s[0][t] = a0;
    s[1][t] = a1;
    s[2][t] = a2;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (t < w)
            for (int a = 0; a < 3; ++a) s[a][t] += s[a][t + w];
        __syncthreads();
    }
    if (t < 3) out[3 * blockIdx.x + t] = s[t][0];
}

}  // namespace

cudaError_t launch_validate_types(const uint8_t* types, size_t N, int* bad, cudaStream_t s) {
    k_validate_types<<<(unsigned)((N + 255) / 256), 256, 0, s>>>(types, N, bad);
    return cudaGetLastError();
}

cudaError_t launch_classify(const Params& p, const uint8_t* types, uint8_t* flags, uint32_t* mask,
                            uint32_t* count, dim3 grid, dim3 block, cudaStream_t s) {
    k_classify<<<grid, block, 0, s>>>(p, types, flags, mask, count);
    return cudaGetLastError();
}

cudaError_t launch_list_special(const Params& p, const uint8_t* flags, uint32_t* list,
                                uint32_t* count, dim3 grid, dim3 block, cudaStream_t s) {
    k_list_special<<<grid, block, 0, s>>>(p, flags, list, count);
    return cudaGetLastError();
}

cudaError_t launch_force_finalize(const double* partial, size_t nblocks, double* stage,
                                  double* out, cudaStream_t s) {
    const size_t chunk = (nblocks + kForceStage - 1) / kForceStage;
    k_force_sum<<<kForceStage, 256, 0, s>>>(partial, nblocks, chunk > 0 ? chunk : 1, stage);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_force_sum<<<1, 256, 0, s>>>(stage, kForceStage, kForceStage, out);
    return cudaGetLastError();
}

}  // namespace lbm
