// Momentum-exchange force of one collision of a caller-held state, computed without allocating
// any device memory.
//
// Some callers cannot call cudaMalloc: plug-ins whose host application owns all device memory
// through its own pool (an allocation behind the pool's back can fail or break its accounting),
// and tools that must not grow the footprint of a process they are embedded in.  This entry point
// serves them: the only working memory it uses is g_noalloc_scratch below, a fixed-size array in
// the library's static device memory, which every GPU that loads the library holds until the
// process exits.  The caller passes the state, the flags and the output.
#include <cmath>
#include <cstdarg>
#include <mutex>

#include "lbm.h"
#include "lbm_kernels.cuh"
#include "lbm_launch.h"

using namespace lbm;

namespace {

// Scratch layout (doubles): [per-block partial sums: 3 per block, kMaxBlocks blocks]
//                           [first-stage sums: 3 x kForceStage] [result: 3] [error word]
constexpr unsigned kThreads = 256;
constexpr unsigned kMaxBlocks = 65536;
constexpr size_t kMaxCells = (size_t)kMaxBlocks * kThreads;  // 16,777,216 cells (256^3)
constexpr size_t kPartialDoubles = 3 * (size_t)kMaxBlocks;
constexpr size_t kStageDoubles = 3 * (size_t)kForceStage;
constexpr size_t kScratchDoubles = kPartialDoubles + kStageDoubles + 4;

__device__ __align__(256) double g_noalloc_scratch[kScratchDoubles];  // 1.5 MiB per device

constexpr int kMaxDevices = 64;
double* g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device
std::mutex g_scratch_mutex;

// Host code cannot use g_noalloc_scratch's name as a device address: look the address up once
// per device, with that device current.
cudaError_t scratch_for_current_device(double** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<double*>(ptr);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

int lbm_noalloc_fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    set_last_error_v(fmt, ap);
    va_end(ap);
    return code;
}

// True when p is device (or managed) memory of device `dev`.
bool is_memory_of_device(const void* p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// One thread per cell: collide the natural state of a FLUID cell (shifted as the step kernels
// store it) and add 2 c_q f*_q for every link q whose partner x + c_q (wrapped, or clamped at an
// OPEN face) is SOLID.  Flag values other than 0, 1, 2 set the error word.
template <bool BODY>
__global__ void __launch_bounds__(kThreads) k_force_of_state(Params p, const float* f,
                                                             const uint8_t* types, double* partial,
                                                             double* error_word) {
    const size_t n = (size_t)blockIdx.x * kThreads + threadIdx.x;
    float fx = 0.f, fy = 0.f, fz = 0.f;
    if (n < p.N) {
        const uint8_t t = types[n];
        if (t > T_INLET) *error_word = 1.0;
        if (t == T_FLUID) {
            const int x = (int)(n % (size_t)p.nx);
            const int y = (int)((n / (size_t)p.nx) % (size_t)p.ny);
            const int z = (int)(n / ((size_t)p.nx * (size_t)p.ny));
            float h[19];
#pragma unroll
            for (int q = 0; q < 19; ++q) h[q] = f[(size_t)q * p.N + n] - wq(q);
            collide<BODY>(h, p);
            uint32_t m = 0;
            for (int q = 1; q < 19; ++q) {
                const Link s = link_cell(p, x, y, z, cx(q), cy(q), cz(q));
                if (types[s.cell] == T_SOLID) m |= 1u << q;
            }
            mask_forces(m, h, fx, fy, fz);
        }
    }
    block_force(fx, fy, fz, partial);
}

}  // namespace

extern "C" int lbm_force_momentum_exchange_noalloc(const float* f, const uint8_t* flags, int nx,
                                                   int ny, int nz, int face_x, int face_y,
                                                   int face_z, float tau, float gx, float gy,
                                                   float gz, double F[3], void* cuda_stream) {
    // argument checks first: no CUDA call is made for a rejected request
    if (!f || !flags || !F)
        return lbm_noalloc_fail(LBM_EINVAL, "lbm_force_momentum_exchange_noalloc: NULL argument");
    if (nx < 1 || ny < 1 || nz < 1)
        return lbm_noalloc_fail(LBM_EINVAL, "lbm_force_momentum_exchange_noalloc: every extent must be >= 1");
    const size_t N = (size_t)nx * (size_t)ny * (size_t)nz;
    if (N > kMaxCells)
        return lbm_noalloc_fail(LBM_EINVAL,
                                "lbm_force_momentum_exchange_noalloc: %zu cells exceed the fixed "
                                "scratch limit of %zu cells (use lbm_force_momentum_exchange)",
                                N, kMaxCells);
    const int faces[3] = {face_x, face_y, face_z};
    const int ext[3] = {nx, ny, nz};
    for (int a = 0; a < 3; ++a)
        if ((faces[a] != LBM_PERIODIC && faces[a] != LBM_OPEN) || (faces[a] == LBM_OPEN && ext[a] < 2))
            return lbm_noalloc_fail(LBM_EINVAL, "lbm_force_momentum_exchange_noalloc: bad face type on axis %d", a);
    if (!std::isfinite(tau) || !(tau > 0.5f))
        return lbm_noalloc_fail(LBM_EINVAL, "lbm_force_momentum_exchange_noalloc: need a finite tau > 1/2");
    if (!std::isfinite(gx) || !std::isfinite(gy) || !std::isfinite(gz))
        return lbm_noalloc_fail(LBM_EINVAL, "lbm_force_momentum_exchange_noalloc: g must be finite");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return lbm_noalloc_fail(LBM_ECUDA, "lbm_force_momentum_exchange_noalloc: no current device");
    }
    if (!is_memory_of_device(f, dev) || !is_memory_of_device(flags, dev))
        return lbm_noalloc_fail(LBM_EINVAL,
                                "lbm_force_momentum_exchange_noalloc: f and flags must be device "
                                "memory of the current device %d (this entry point cannot stage "
                                "host data or reach another device's memory)", dev);

    double* scratch = nullptr;
    cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess)
        return lbm_noalloc_fail(LBM_ECUDA, "lbm_force_momentum_exchange_noalloc: scratch address: %s",
                                cudaGetErrorString(e));
    double* partial = scratch;
    double* stage = scratch + kPartialDoubles;
    double* result_dev = stage + kStageDoubles;
    double* error_word = result_dev + 3;
    cudaStream_t s = (cudaStream_t)cuda_stream;

    Params p{};
    p.nx = nx;
    p.ny = ny;
    p.nz = nz;
    p.N = N;
    for (int a = 0; a < 3; ++a) p.open[a] = faces[a] == LBM_OPEN;
    p.omega = 1.0f / tau;
    p.g[0] = gx;
    p.g[1] = gy;
    p.g[2] = gz;
    guo_constants(tau, p.g, p.tau_g, p.wk);
    const bool body = gx != 0.f || gy != 0.f || gz != 0.f;
    const unsigned blocks = (unsigned)((N + kThreads - 1) / kThreads);

    // the error word is the only scratch value read before this call writes it
    e = cudaMemsetAsync(error_word, 0, sizeof(double), s);
    if (e == cudaSuccess) {
        if (body) k_force_of_state<true><<<blocks, kThreads, 0, s>>>(p, f, flags, partial, error_word);
        else k_force_of_state<false><<<blocks, kThreads, 0, s>>>(p, f, flags, partial, error_word);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_force_finalize(partial, blocks, stage, result_dev, s);
    double result[4] = {0.0, 0.0, 0.0, 0.0};
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(result, result_dev, 3 * sizeof(double), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(result + 3, error_word, sizeof(double), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return lbm_noalloc_fail(LBM_ECUDA, "lbm_force_momentum_exchange_noalloc: %s", cudaGetErrorString(e));
    if (result[3] != 0.0)
        return lbm_noalloc_fail(LBM_EINVAL,
                                "lbm_force_momentum_exchange_noalloc: flag values must be 0, 1 or 2");
    for (int a = 0; a < 3; ++a) F[a] = result[a];
    return LBM_OK;
}
