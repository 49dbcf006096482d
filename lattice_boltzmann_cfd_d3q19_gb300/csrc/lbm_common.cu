// Layout-independent kernels: flag validation and classification, force finalisation.
#include "lbm_kernels.cuh"
#include "lbm_launch.h"

namespace lbm {
namespace {

__global__ void __launch_bounds__(256) k_validate_types(const uint8_t* types, size_t N, int* bad) {
    const size_t n = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n < N && types[n] > T_INLET) *bad = 1;
}

// flags = type | F_BULK when the cell is FLUID and all 18 neighbours are inside the domain
// (wrapped on periodic axes, not beyond an open face) and FLUID.
__global__ void __launch_bounds__(256) k_classify(Params p, const uint8_t* types, uint8_t* flags) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= p.nx || y >= p.ny) return;
    const uint32_t n = (uint32_t)x + (uint32_t)p.nx * ((uint32_t)y + (uint32_t)p.ny * z);
    const uint8_t t = types[n];
    uint8_t out = t;
    if (t == T_FLUID) {
        bool bulk = true;
        for (int q = 1; q < 19; ++q) {
            const Link s = link_cell(p, x, y, z, cx(q), cy(q), cz(q));
            if (s.face >= 0 || types[s.cell] != T_FLUID) bulk = false;
        }
        if (bulk) out |= F_BULK;
    }
    flags[n] = out;
}

// Sums the per-block partials in a fixed order (strided per thread, then a tree), in fp64.
__global__ void __launch_bounds__(256) k_force_finalize(const double* partial, size_t nblocks,
                                                        double* out) {
    __shared__ double s[3][256];
    const int t = threadIdx.x;
    double a0 = 0.0, a1 = 0.0, a2 = 0.0;
    for (size_t b = t; b < nblocks; b += 256) {
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
    if (t < 3) out[t] = s[t][0];
}

}  // namespace

cudaError_t launch_validate_types(const uint8_t* types, size_t N, int* bad, cudaStream_t s) {
    k_validate_types<<<(unsigned)((N + 255) / 256), 256, 0, s>>>(types, N, bad);
    return cudaGetLastError();
}

cudaError_t launch_classify(const Params& p, const uint8_t* types, uint8_t* flags, dim3 grid,
                            dim3 block, cudaStream_t s) {
    k_classify<<<grid, block, 0, s>>>(p, types, flags);
    return cudaGetLastError();
}

cudaError_t launch_force_finalize(const double* partial, size_t nblocks, double* out,
                                  cudaStream_t s) {
    k_force_finalize<<<1, 256, 0, s>>>(partial, nblocks, out);
    return cudaGetLastError();
}

}  // namespace lbm
