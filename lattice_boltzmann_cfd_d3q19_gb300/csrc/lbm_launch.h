// Host-side launch interface between the C ABI and the layout-specific kernel instantiations.
#pragma once

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "lbm_device.cuh"

namespace lbm {

// kernel kinds (also the profiling kinds of the C ABI)
enum : int {
    K_AA_EVEN = 0,
    K_AA_ODD = 1,
    K_AB_PULL = 2,
    K_AB_COLLIDE = 3,
    K_STREAM = 4,
    K_PREGATHER = 5,
    K_FORCE = 6,
    K_BOUNDARY = 7,  // special-cell kernels of the AA odd, A-B pull and streaming steps
    K_NUM_KINDS = 8
};

struct LayoutOps {
    // step kernels: K_AA_EVEN, K_AA_ODD, K_AB_PULL, K_AB_COLLIDE, K_STREAM
    cudaError_t (*cells)(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                         cudaStream_t s);
    // two-cell step kernels (K_AA_EVEN, K_AA_ODD, K_AB_PULL, K_AB_COLLIDE) for the stream layouts
    // on grids with an even nx and 19 N <= 2^32, launched over cell pairs; cudaErrorNotSupported
    // for the other layouts
    cudaError_t (*cells2)(int kind, const Params& p, bool force, bool body, dim3 grid, dim3 block,
                          cudaStream_t s);
    // AA odd step with the gather staged by TMA bulk copies (stream layouts, 16 | nx <= 512,
    // 19 N <= 2^32): `grid` persistent CTAs of 256 threads; cudaErrorNotSupported otherwise
    cudaError_t (*odd_tma)(const Params& p, bool force, bool body, unsigned grid, cudaStream_t s);
    // A-B pull of the collision layout with its gather staged in 2.5D tiles (32 | nx,
    // 19 N <= 2^32): `grid` = (nx / 32, ceil(ny / 8), z chunks) blocks of 256 threads;
    // cudaErrorNotSupported for the other layouts.  tile_prepare raises the kernel's dynamic
    // shared-memory limit on the current device (a no-op for the other layouts).
    cudaError_t (*ab_pull_tile)(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s);
    // AA odd step of the collision layout in 2.5D tiles, updated in place in shared memory (32 | nx,
    // ny >= 10, 19 N <= 2^32; the same grid); cudaErrorNotSupported for the other layouts
    cudaError_t (*aa_odd_tile)(const Params& p, bool force, bool body, dim3 grid, cudaStream_t s);
    cudaError_t (*tile_prepare)();
    // boundary kernel over the special-cell list for main kind K_AA_ODD, K_AB_PULL or K_STREAM
    cudaError_t (*special)(int kind, const Params& p, bool force, bool body, cudaStream_t s);
    // open-face pre-gather of the AA odd step, every open face in one launch
    cudaError_t (*pregather)(const Params& p, cudaStream_t s);
    cudaError_t (*pack)(const Params& p, const float* in, size_t i0, size_t count, cudaStream_t s);
    cudaError_t (*unpack)(const Params& p, int state, float* out, size_t i0, size_t count,
                          cudaStream_t s);
    cudaError_t (*equilibrium)(const Params& p, const float* rho, const float* u0, const float* u1,
                               const float* u2, uint32_t n0, uint32_t count, cudaStream_t s);
    cudaError_t (*macro)(const Params& p, int state, const float inlet[4], float* rho, float* u0,
                         float* u1, float* u2, uint32_t n0, uint32_t count, cudaStream_t s);
    cudaError_t (*check_finite)(const Params& p, int* bad, dim3 grid, dim3 block, cudaStream_t s);
    // the INLET cells' post-collision slots of a buffer in state ST_POST_AA or ST_POST_AB set to
    // the reservoir's f_eq(rho_in, u_in)
    cudaError_t (*fill_inlet)(const Params& p, int state, dim3 grid, dim3 block, cudaStream_t s);
    // slab halos of the A-B post-collision state: the c_z = -1 populations of plane 1 into lo and
    // the c_z = +1 ones of plane nz - 2 into hi; the reverse into the ghost planes 0 and nz - 1
    cudaError_t (*halo_pack)(const Params& p, void* lo, void* hi, cudaStream_t s);
    cudaError_t (*halo_unpack)(const Params& p, const void* below, const void* above, cudaStream_t s);
};

const LayoutOps& layout_ops_stream();
const LayoutOps& layout_ops_bundle();
const LayoutOps& layout_ops_collision();
const LayoutOps& layout_ops_stream_fp16();

// layout-independent kernels
cudaError_t launch_validate_types(const uint8_t* types, size_t N, int* bad, cudaStream_t s);
// flags, solid-link masks and the number of special cells (added to *count)
cudaError_t launch_classify(const Params& p, const uint8_t* types, uint8_t* flags, uint32_t* mask,
                            uint32_t* count, dim3 grid, dim3 block, cudaStream_t s);
// appends the index of every special cell to list (order unspecified), *count as the cursor
cudaError_t launch_list_special(const Params& p, const uint8_t* flags, uint32_t* list,
                                uint32_t* count, dim3 grid, dim3 block, cudaStream_t s);
// fixed-order fp64 sum of nblocks partial triples: per-chunk sums into stage (kForceStage
// triples), then one block -> out[3].  Two launches.
constexpr unsigned kForceStage = 256;
cudaError_t launch_force_finalize(const double* partial, size_t nblocks, double* stage,
                                  double* out, cudaStream_t s);

// Launch constants of the Guo forcing for relaxation time tau and body acceleration g.
void guo_constants(float tau, const float g[3], float tau_g[3], float wk[19]);

// Sets the calling thread's lbm_last_error() message (printf-style).
void set_last_error_v(const char* fmt, va_list ap);

}  // namespace lbm
