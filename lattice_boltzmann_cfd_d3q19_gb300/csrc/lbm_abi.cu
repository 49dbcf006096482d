// C ABI of the D3Q19 BGK library: context, buffers, the step sequence and host/device transfers.
// The arithmetic lives in the kernels (lbm_kernels.cuh); this file only validates arguments,
// owns device memory and enqueues launches on the context's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "lbm.h"
#include "lbm_launch.h"

using namespace lbm;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    if (e == cudaErrorMemoryAllocation)
        return fail(LBM_ENOMEM, "%s: out of device memory (%s)", what, cudaGetErrorString(e));
    return fail(LBM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define LBM_CUDA(call, what)                                  \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(e_, (what));  \
    } while (0)

bool is_device_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// f_eq(rho, u) - w in double, rounded once (host-side inlet constant).
void shifted_equilibrium(double rho, const double u[3], float out[19]) {
    const double uu = u[0] * u[0] + u[1] * u[1] + u[2] * u[2];
    for (int q = 0; q < 19; ++q) {
        const double cu = cx(q) * u[0] + cy(q) * u[1] + cz(q) * u[2];
        const double w = q == 0 ? 1.0 / 3.0 : q <= 6 ? 1.0 / 18.0 : 1.0 / 36.0;
        out[q] = (float)(w * (rho - 1.0 + rho * (3.0 * cu + 4.5 * cu * cu - 1.5 * uu)));
    }
}

constexpr size_t kStagingFloats = size_t(32) << 20;  // 128 MiB host-transfer staging

}  // namespace

// Launch constants of the Guo forcing as the collision applies it (see collide() in
// lbm_device.cuh): the equilibrium velocity shift tau g and, per population,
// -omega (tau - 1/2)^2 w_q (4.5 (c_q.g)^2 - 1.5 g.g); computed in double, rounded once.
void lbm::guo_constants(float tau, const float g[3], float tau_g[3], float wk[19]) {
    const double t = tau, om = 1.0 / t, a = t - 0.5;
    const double gg = (double)g[0] * g[0] + (double)g[1] * g[1] + (double)g[2] * g[2];
    for (int k = 0; k < 3; ++k) tau_g[k] = (float)(t * g[k]);
    for (int q = 0; q < 19; ++q) {
        const double cg = cx(q) * (double)g[0] + cy(q) * (double)g[1] + cz(q) * (double)g[2];
        const double w = q == 0 ? 1.0 / 3.0 : q <= 6 ? 1.0 / 18.0 : 1.0 / 36.0;
        wk[q] = (float)(-om * a * a * w * (4.5 * cg * cg - 1.5 * gg));
    }
}

namespace {

}  // namespace

void lbm::set_last_error_v(const char* fmt, va_list ap) {
    char buf[512];
    vsnprintf(buf, sizeof buf, fmt, ap);
    g_err = buf;
}

struct lbm_ctx {
    int n[3] = {0, 0, 0};
    size_t N = 0;
    float tau = 0.f, omega = 0.f;
    int layout = 0, streaming = 0;
    const LayoutOps* ops = nullptr;
    int face[3] = {LBM_PERIODIC, LBM_PERIODIC, LBM_PERIODIC};
    float g[3] = {0.f, 0.f, 0.f};
    float inlet[4] = {1.f, 0.f, 0.f, 0.f};
    float heq_in[19] = {};
    void* buf[2] = {nullptr, nullptr};
    int cur = 0;
    int state = ST_NATURAL;
    uint8_t* types = nullptr;
    uint8_t* flags = nullptr;
    uint32_t* mask = nullptr;
    uint32_t* special = nullptr;  // sorted indices of the special FLUID cells
    uint32_t n_special = 0;
    // with ghost planes: the special cells of plane 1 are special[0, sp_lo_end), those of plane
    // nz - 2 special[sp_hi_begin, n_special) (the list is sorted, ghost cells are never special)
    uint32_t sp_lo_end = 0, sp_hi_begin = 0;
    bool split = false;           // a slab step is open (lbm_slab_step_begin without its end)
    uint32_t* count_dev = nullptr;  // counters: special cells, SOLID links, MOVING_WALL links, INLET cells
    int any_solid_link = 0;
    int any_moving = 0;
    int any_inlet = 0;
    float uw[3] = {0.f, 0.f, 0.f};
    float* scratch = nullptr;
    size_t face_base[3][2] = {};
    double* partial = nullptr;    // nblocks main-kernel partials, then the boundary kernels'
    size_t partial_cap = 0;       // triples allocated
    size_t nblocks = 0;
    // two-cell kernels: launch geometry over cell pairs, and whether the caller allows them
    dim3 grid2, block2;
    size_t nblocks2 = 0;
    bool pairs_allowed = true;
    // TMA-staged AA odd kernel: persistent grid and whether the caller allows it
    unsigned ntma = 0;
    // 2.5D-tiled A-B pull of the collision layout: its grid (z chunks of the tiles) and blocks
    dim3 tile_grid;
    size_t ntile = 0;
    bool tma_allowed = false;  // opt-in: measured slower than the register kernels
    int* fault_dev = nullptr;   // set by a kernel whose bounded wait ran out (sticky)
    // test hook (LBM_TEST_STAGE_TIMEOUT=1 at lbm_create): the staged kernel announces 16 bytes
    // more than it copies, so its first wait runs out; nothing faults
    uint32_t extra_tx = 0;
    bool ghost = false;           // z = 0 and z = nz - 1 are ghost planes of a slab decomposition
    int* fault_host = nullptr;
    size_t force_triples = 0;     // partial triples written by the step that computes the force
    double* stage = nullptr;
    double* force_dev = nullptr;
    double* force_host = nullptr;
    int* err_dev = nullptr;
    int* err_host = nullptr;
    float* staging = nullptr;
    // double-buffered host transfers: the copy of one half of the staging buffer (on the private
    // copy stream) overlaps the kernel on the other half (on the context stream)
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t stage_full[2] = {nullptr, nullptr};  // a half holds data for its consumer
    cudaEvent_t stage_free[2] = {nullptr, nullptr};  // a half's consumer is done with it
    cudaEvent_t stage_mark = nullptr;                // start / end marker between the streams
    cudaStream_t stream = nullptr;
    // The boundary kernel of a step runs beside the step's main kernel, on a second stream of the
    // highest priority forked from `stream` and joined back into it, where the main kernel
    // stores into no slot of a special cell (the AA odd kernels, the one-cell A-B pull and the
    // streaming pass): the special cells' latency-bound warps then overlap the main kernel's
    // streaming instead of following it.  The two-cell A-B pull and the staged pull of the bundle
    // and collision layouts write special cells' slots with their whole-sector stores and keep
    // the serial order.  Serial while profiling
    // (per-kernel times) or when the caller switches it off.
    cudaStream_t side_stream = nullptr;
    cudaEvent_t side_fork = nullptr, side_join = nullptr;
    bool overlap_allowed = true;
    bool overlap(int kind) const {
        if (!overlap_allowed || profiling || n_special == 0) return false;
        // the two-cell pull and the staged pull of the non-SoA layouts write special cells' slots,
        // and so does the tiled odd step (whole records)
        if (kind == K_AA_ODD && tiled_odd()) return false;
        return !(kind == K_AB_PULL && (pairs() || !is_soa(layout)));
    }
    int64_t steps = 0;
    bool force_valid = false;
    int64_t launches = 0;
    dim3 grid, block;
    bool profiling = false;
    // CUDA graphs of step sequences, captured on a private stream and launched on `stream`
    struct GraphEntry {
        int len, state, cur, force;
        cudaGraphExec_t exec;
        int64_t kernels;  // kernel launches one replay performs
    };
    bool use_graphs = true;
    cudaStream_t capture_stream = nullptr;
    std::vector<GraphEntry> graphs;
    void drop_graphs() {
        for (auto& g : graphs) cudaGraphExecDestroy(g.exec);
        graphs.clear();
    }
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> prof[K_NUM_KINDS];
    std::vector<cudaEvent_t> event_pool;

    Params params(void* A, void* B) const {
        Params p;
        p.A = A;
        p.B = B;
        p.flags = flags;
        p.mask = mask;
        p.any_solid_link = any_solid_link;
        p.any_moving = any_moving;
        p.any_inlet = any_inlet;
        p.open_special = streaming == LBM_STREAMING_AA;
        p.ghost_z = ghost ? 1 : 0;
        for (int a = 0; a < 3; ++a) p.uw[a] = uw[a];
        for (int q = 0; q < 19; ++q) {
            const double w = q == 0 ? 1.0 / 3.0 : q <= 6 ? 1.0 / 18.0 : 1.0 / 36.0;
            p.wterm[q] = (float)(6.0 * w * (cx(q) * (double)uw[0] + cy(q) * (double)uw[1] +
                                            cz(q) * (double)uw[2]));
        }
        p.special = special;
        p.n_special = n_special;
        p.scratch = scratch;
        p.partial = partial;
        p.fault = fault_dev;
        p.zrev = 0;
        p.zbase = 0;
        p.zstep = 1;
        p.part_main = 0;
        p.extra_tx = extra_tx;
        p.part_special = main_blocks() * kWarpsPerBlock;
        p.nx = n[0];
        p.ny = n[1];
        p.nz = n[2];
        for (int a = 0; a < 3; ++a) p.open[a] = face[a] == LBM_OPEN;
        p.N = N;
        for (int a = 0; a < 3; ++a)
            for (int s = 0; s < 2; ++s) p.face_base[a][s] = face_base[a][s];
        p.omega = omega;
        for (int a = 0; a < 3; ++a) p.g[a] = g[a];
        guo_constants(tau, g, p.tau_g, p.wk);
        for (int q = 0; q < 19; ++q) p.heq_in[q] = heq_in[q];
        for (int q = 0; q < 19; ++q) {
            const size_t off = plane_offset(q), off_opp = plane_offset(opp(q));
            const size_t bytes = off * elem_bytes_of();
            p.pa[q] = A ? static_cast<char*>(A) + bytes : nullptr;
            p.pb[q] = B ? static_cast<char*>(B) + bytes : nullptr;
            p.pdiff[q] = (long long)off - (long long)off_opp;
            p.plane32[q] = (uint32_t)off;  // used only while 19 N <= 2^32
        }
        return p;
    }
    // element offset of population q of cell 0 in the population layout
    size_t plane_offset(int q) const {
        switch (layout) {
            case LBM_LAYOUT_BUNDLE: return idx<LAYOUT_BUNDLE>(q, 0, N);
            case LBM_LAYOUT_COLLISION: return idx<LAYOUT_COLLISION>(q, 0, N);
            case LBM_LAYOUT_STREAM_FP16: return idx<LAYOUT_STREAM_FP16>(q, 0, N);
            default: return idx<LAYOUT_STREAM>(q, 0, N);
        }
    }
    // the hot step kernels run two cells per thread: stream layouts, even nx, 32-bit offsets
    bool pairs() const {
        return pairs_allowed && is_soa(layout) && n[0] % 2 == 0 && 19 * N <= (size_t(1) << 32);
    }
    // the AA odd step stages its gather through shared memory (TMA bulk copies of whole rows)
    bool tma() const { return pairs() && tma_allowed && n[0] % 16 == 0 && n[0] <= 512 && ntma > 0; }
    // the collision layout's A-B pull stages its gather in 2.5D tiles
    bool tiled() const {
        return layout == LBM_LAYOUT_COLLISION && n[0] % kTileX == 0 && 19 * N <= (size_t(1) << 32) &&
               ntile > 0;
    }
    // and its AA odd step runs in the same tiles, in place in shared memory, where no two rows of a
    // halo tile are one row of the grid
    bool tiled_odd() const { return tiled() && n[1] >= kTileY + 2; }
    // blocks of the step kernels that write force partials (the boundary kernels' partials follow)
    size_t main_blocks() const { return pairs() || bundle_pairs() ? nblocks2 : nblocks; }
    // the bundle layout's AA even step also runs two cells per thread (aligned pair runs)
    bool bundle_pairs() const {
        return pairs_allowed && layout == LBM_LAYOUT_BUNDLE && n[0] % 2 == 0 &&
               19 * N <= (size_t(1) << 32);
    }
    // kernels launched over cell pairs for step kind `kind`
    bool pairs_for(int kind) const {
        if (kind == K_STREAM) return false;
        return pairs() || bundle_pairs();
    }
    size_t main_blocks_for(int kind) const {
        if (kind == K_AA_ODD && tma()) return ntma;
        if (kind == K_AB_PULL && tiled()) return ntile;
        if (kind == K_AA_ODD && tiled_odd()) return ntile;
        return pairs_for(kind) ? nblocks2 : nblocks;
    }
    bool body() const { return g[0] != 0.f || g[1] != 0.f || g[2] != 0.f; }
    bool any_open() const { return face[0] == LBM_OPEN || face[1] == LBM_OPEN || face[2] == LBM_OPEN; }
    // buffer holding the current state and its meaning
    void* state_buffer() const { return streaming == LBM_STREAMING_AA ? buf[0] : buf[cur]; }
    size_t elem_bytes_of() const { return layout == LBM_LAYOUT_STREAM_FP16 ? 2 : 4; }

    cudaEvent_t take_event() {
        cudaEvent_t e = nullptr;
        if (!event_pool.empty()) {
            e = event_pool.back();
            event_pool.pop_back();
        } else if (cudaEventCreate(&e) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return e;
    }
    void release_profile() {
        for (auto& v : prof) {
            for (auto& pr : v) {
                event_pool.push_back(pr.first);
                event_pool.push_back(pr.second);
            }
            v.clear();
        }
    }
    void free_all() {
        if (stream) cudaStreamSynchronize(stream);
        drop_graphs();
        if (capture_stream) cudaStreamDestroy(capture_stream);
        release_profile();
        for (cudaEvent_t e : event_pool) cudaEventDestroy(e);
        event_pool.clear();
        cudaFree(buf[0]);
        cudaFree(buf[1]);
        cudaFree(types);
        cudaFree(flags);
        cudaFree(mask);
        cudaFree(special);
        cudaFree(count_dev);
        cudaFree(stage);
        cudaFree(scratch);
        cudaFree(partial);
        cudaFree(force_dev);
        cudaFree(err_dev);
        cudaFree(staging);
        for (int h = 0; h < 2; ++h) {
            if (stage_full[h]) cudaEventDestroy(stage_full[h]);
            if (stage_free[h]) cudaEventDestroy(stage_free[h]);
        }
        if (stage_mark) cudaEventDestroy(stage_mark);
        if (copy_stream) cudaStreamDestroy(copy_stream);
        if (side_fork) cudaEventDestroy(side_fork);
        if (side_join) cudaEventDestroy(side_join);
        if (side_stream) cudaStreamDestroy(side_stream);
        cudaFreeHost(force_host);
        cudaFreeHost(err_host);
        cudaFree(fault_dev);
        cudaFreeHost(fault_host);
    }
};

namespace {

const LayoutOps* ops_for(int layout) {
    switch (layout) {
        case LBM_LAYOUT_STREAM: return &layout_ops_stream();
        case LBM_LAYOUT_BUNDLE: return &layout_ops_bundle();
        case LBM_LAYOUT_COLLISION: return &layout_ops_collision();
        case LBM_LAYOUT_STREAM_FP16: return &layout_ops_stream_fp16();
    }
    return nullptr;
}

int ensure_staging(lbm_ctx* c) {
    if (!c->staging) LBM_CUDA(cudaMalloc(&c->staging, kStagingFloats * sizeof(float)), "staging buffer");
    if (!c->copy_stream)
        LBM_CUDA(cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking), "copy stream");
    for (int h = 0; h < 2; ++h) {
        if (!c->stage_full[h])
            LBM_CUDA(cudaEventCreateWithFlags(&c->stage_full[h], cudaEventDisableTiming), "staging events");
        if (!c->stage_free[h])
            LBM_CUDA(cudaEventCreateWithFlags(&c->stage_free[h], cudaEventDisableTiming), "staging events");
    }
    if (!c->stage_mark)
        LBM_CUDA(cudaEventCreateWithFlags(&c->stage_mark, cudaEventDisableTiming), "staging events");
    // the copy stream starts after the work already on the context stream
    LBM_CUDA(cudaEventRecord(c->stage_mark, c->stream), "staging");
    LBM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->stage_mark, 0), "staging");
    return LBM_OK;
}

constexpr size_t kStageHalf = kStagingFloats / 2;  // floats per staging half

// host -> staging half h (copy stream), then `use` it on the context stream
int stage_in(lbm_ctx* c, int h, float* dst_half, const float* src, size_t count) {
    LBM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->stage_free[h], 0), "staging");
    LBM_CUDA(cudaMemcpyAsync(dst_half, src, count * sizeof(float), cudaMemcpyDefault, c->copy_stream),
             "host copy");
    return LBM_OK;
}
int stage_in_done(lbm_ctx* c, int h) {
    LBM_CUDA(cudaEventRecord(c->stage_full[h], c->copy_stream), "staging");
    LBM_CUDA(cudaStreamWaitEvent(c->stream, c->stage_full[h], 0), "staging");
    return LBM_OK;
}
// after the context stream's kernel has read (upload) or written (read-back) half h
int stage_used(lbm_ctx* c, int h) {
    LBM_CUDA(cudaEventRecord(c->stage_free[h], c->stream), "staging");
    return LBM_OK;
}
// read-back: the context stream wrote half h; copy it to the host on the copy stream
int stage_out(lbm_ctx* c, int h, float* dst, const float* src_half, size_t count) {
    LBM_CUDA(cudaMemcpyAsync(dst, src_half, count * sizeof(float), cudaMemcpyDefault, c->copy_stream),
             "host copy");
    return LBM_OK;
}
int stage_out_begin(lbm_ctx* c, int h) {
    // the copy that last read half h is done before the kernel overwrites it
    LBM_CUDA(cudaStreamWaitEvent(c->stream, c->stage_free[h], 0), "staging");
    return LBM_OK;
}
int stage_out_ready(lbm_ctx* c, int h) {
    LBM_CUDA(cudaEventRecord(c->stage_full[h], c->stream), "staging");
    LBM_CUDA(cudaStreamWaitEvent(c->copy_stream, c->stage_full[h], 0), "staging");
    return LBM_OK;
}
int stage_out_copied(lbm_ctx* c, int h) {
    LBM_CUDA(cudaEventRecord(c->stage_free[h], c->copy_stream), "staging");
    return LBM_OK;
}
// the context stream completes after every copy of the copy stream
int stage_end(lbm_ctx* c) {
    LBM_CUDA(cudaEventRecord(c->stage_mark, c->copy_stream), "staging");
    LBM_CUDA(cudaStreamWaitEvent(c->stream, c->stage_mark, 0), "staging");
    return LBM_OK;
}

// blocks of the boundary kernels that write force partials: one warp per special cell
unsigned special_blocks(uint32_t n_special) { return (n_special + 7) / 8; }

// one fp64 partial triple per warp of the step kernels and of the boundary kernels
size_t partial_triples(size_t main_blocks, uint32_t n_special) {
    return (main_blocks + special_blocks(n_special)) * kWarpsPerBlock;
}

// Recompute flags, solid-link masks and the sorted special-cell list from the cell types and
// faces.  Synchronous.
int classify(lbm_ctx* c) {
    Params p = c->params(nullptr, nullptr);
    LBM_CUDA(cudaMemsetAsync(c->count_dev, 0, 4 * sizeof(uint32_t), c->stream), "classify");
    LBM_CUDA(launch_classify(p, c->types, c->flags, c->mask, c->count_dev, c->grid, c->block,
                             c->stream), "classify flags");
    ++c->launches;
    uint32_t counts[4] = {0, 0, 0, 0};
    LBM_CUDA(cudaMemcpyAsync(counts, c->count_dev, 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost,
                             c->stream), "classify");
    LBM_CUDA(cudaStreamSynchronize(c->stream), "classify");
    const uint32_t count = counts[0];
    std::vector<uint32_t> list(count);
    uint32_t* dev_list = nullptr;
    if (count > 0) {
        LBM_CUDA(cudaMalloc(&dev_list, count * sizeof(uint32_t)), "classify: special-cell list");
        cudaError_t e = cudaMemsetAsync(c->count_dev, 0, sizeof(uint32_t), c->stream);
        if (e == cudaSuccess)
            e = launch_list_special(p, c->flags, dev_list, c->count_dev, c->grid, c->block, c->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(list.data(), dev_list, count * sizeof(uint32_t),
                                cudaMemcpyDeviceToHost, c->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
        if (e == cudaSuccess) {
            ++c->launches;
            // a fixed cell order keeps the boundary kernels' force partial sums reproducible
            std::sort(list.begin(), list.end());
            e = cudaMemcpyAsync(dev_list, list.data(), count * sizeof(uint32_t),
                                cudaMemcpyHostToDevice, c->stream);
        }
        if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
        if (e != cudaSuccess) {
            cudaFree(dev_list);
            return cuda_fail(e, "classify: special-cell list");
        }
    }
    // one triple per warp of the largest main grid: the one-cell, two-cell, TMA-staged and tiled
    // grids (a thin grid can have more tiles than one-cell blocks)
    const size_t need =
        partial_triples(std::max({c->nblocks, c->nblocks2, (size_t)c->ntma, c->ntile}), count);
    if (need > c->partial_cap) {
        double* np_ = nullptr;
        cudaError_t e = cudaMalloc(&np_, 3 * need * sizeof(double));
        if (e != cudaSuccess) {
            cudaFree(dev_list);
            return cuda_fail(e, "classify: force partials");
        }
        cudaFree(c->partial);
        c->partial = np_;
        c->partial_cap = need;
    }
    cudaFree(c->special);
    c->special = dev_list;
    c->n_special = count;
    {
        const uint32_t area = (uint32_t)c->n[0] * (uint32_t)c->n[1];
        const uint32_t nz = (uint32_t)c->n[2];
        c->sp_lo_end = (uint32_t)(std::lower_bound(list.begin(), list.end(), 2 * area) - list.begin());
        c->sp_hi_begin = nz >= 3 ? (uint32_t)(std::lower_bound(list.begin(), list.end(), (nz - 2) * area) -
                                             list.begin())
                                 : count;
    }
    c->any_solid_link = counts[1] > 0;
    c->any_moving = counts[2] > 0;
    c->any_inlet = counts[3] > 0;
    return LBM_OK;
}

// Sweep direction of a step kernel: each step walks the z planes opposite to the step before, so
// it starts on the planes the previous step wrote last (still in L2 on grids near its size).
int z_reversed(const lbm_ctx* c, int kind) {
    switch (kind) {
        // the tiled odd step runs its chunks of planes upwards, so the even step after it goes down
        case K_AA_EVEN: return c->tiled_odd() ? 1 : 0;
        case K_AA_ODD: return 1;
        case K_AB_PULL: return c->cur;
        case K_STREAM: return 1;
        default: return 0;  // A-B / AB2 collision from the natural state
    }
}

// Launch a step kernel (or, for K_BOUNDARY, the boundary kernel of step kind `main_kind`, on
// `boundary_stream` when given), timed when profiling is on.
int launch_kind(lbm_ctx* c, int kind, const Params& p_in, bool force, int main_kind = -1,
                cudaStream_t boundary_stream = nullptr) {
    Params p = p_in;
    p.zrev = z_reversed(c, kind);
    if (p.zrev) {
        p.zbase = c->n[2] - 1;
        p.zstep = -1;
    }
    if (kind == K_BOUNDARY && c->n_special == 0) return LBM_OK;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (c->profiling) {
        e0 = c->take_event();
        e1 = c->take_event();
        if (e0) cudaEventRecord(e0, c->stream);
    }
    cudaError_t e = cudaSuccess;
    if (kind == K_PREGATHER) {
        e = c->ops->pregather(p, c->stream);
        ++c->launches;
    } else if (kind == K_FORCE) {
        e = launch_force_finalize(c->partial, c->force_triples, c->stage, c->force_dev, c->stream);
        c->launches += 2;
    } else if (kind == K_BOUNDARY) {
        e = c->ops->special(main_kind, p, force, c->body(),
                            boundary_stream ? boundary_stream : c->stream);
        ++c->launches;
        if (force) c->force_triples = partial_triples(c->main_blocks_for(main_kind), c->n_special);
    } else {
        const bool two = c->pairs_for(kind);
        if (kind == K_AA_ODD && c->tma())
            e = c->ops->odd_tma(p, force, c->body(), c->ntma, c->stream);
        else if (kind == K_AB_PULL && c->tiled())
            e = c->ops->ab_pull_tile(p, force, c->body(), c->tile_grid, c->stream);
        else if (kind == K_AA_ODD && c->tiled_odd())
            e = c->ops->aa_odd_tile(p, force, c->body(), c->tile_grid, c->stream);
        else if (two)
            e = c->ops->cells2(kind, p, force, c->body(), c->grid2, c->block2, c->stream);
        else
            e = c->ops->cells(kind, p, force, c->body(), c->grid, c->block, c->stream);
        ++c->launches;
        if (force) c->force_triples = partial_triples(c->main_blocks_for(kind), 0);
    }
    if (c->profiling && e0 && e1) {
        cudaEventRecord(e1, c->stream);
        c->prof[kind].emplace_back(e0, e1);
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return LBM_OK;
}

// The main kernel of step kind `kind` and its boundary kernel: side by side on two streams when
// the context allows it, else one after the other on the context stream.
int main_and_boundary(lbm_ctx* c, int kind, const Params& p, bool force) {
    if (!c->overlap(kind)) {
        int rc = launch_kind(c, kind, p, force);
        if (rc == LBM_OK) rc = launch_kind(c, K_BOUNDARY, p, force, kind);
        return rc;
    }
    LBM_CUDA(cudaEventRecord(c->side_fork, c->stream), "lbm_step: fork");
    LBM_CUDA(cudaStreamWaitEvent(c->side_stream, c->side_fork, 0), "lbm_step: fork");
    // the boundary kernel first: its blocks are then dispatched ahead of the main kernel's
    int rc = launch_kind(c, K_BOUNDARY, p, force, kind, c->side_stream);
    if (rc == LBM_OK) rc = launch_kind(c, kind, p, force);
    // joined even after a failed launch, so that a capture in progress ends joined
    cudaError_t e = cudaEventRecord(c->side_join, c->side_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->stream, c->side_join, 0);
    if (rc != LBM_OK) return rc;
    if (e != cudaSuccess) return cuda_fail(e, "lbm_step: join");
    // both kernels' force partials (the main kernel's launch recorded only its own)
    if (force) c->force_triples = partial_triples(c->main_blocks_for(kind), c->n_special);
    return LBM_OK;
}

int step_once(lbm_ctx* c, bool last) {
    int rc = LBM_OK;
    if (c->streaming == LBM_STREAMING_AA) {
        const Params p = c->params(c->buf[0], c->buf[0]);
        if (c->state == ST_NATURAL) {
            rc = launch_kind(c, K_AA_EVEN, p, last);
            c->state = ST_POST_AA;
        } else {
            // open-face sources are copied before either odd kernel writes
            Params po = p;
            po.part_special = c->main_blocks_for(K_AA_ODD) * kWarpsPerBlock;
            if (c->any_open()) rc = launch_kind(c, K_PREGATHER, po, false);
            if (rc == LBM_OK) rc = main_and_boundary(c, K_AA_ODD, po, last);
            c->state = ST_NATURAL;
        }
    } else if (c->streaming == LBM_STREAMING_AB) {
        const Params p = c->params(c->buf[c->cur], c->buf[c->cur ^ 1]);
        if (c->state == ST_NATURAL) {
            rc = launch_kind(c, K_AB_COLLIDE, p, last);
        } else {
            // the boundary kernel's force partials follow those of the pull's own grid
            Params pp = p;
            pp.part_special = c->main_blocks_for(K_AB_PULL) * kWarpsPerBlock;
            rc = main_and_boundary(c, K_AB_PULL, pp, last);
        }
        c->cur ^= 1;
        c->state = ST_POST_AB;
    } else {  // two-pass: collide in place, then pull into the other buffer
        const Params pc = c->params(c->buf[c->cur], c->buf[c->cur]);
        rc = launch_kind(c, K_AB_COLLIDE, pc, last);
        const Params ps = c->params(c->buf[c->cur], c->buf[c->cur ^ 1]);
        if (rc == LBM_OK) rc = main_and_boundary(c, K_STREAM, ps, false);
        c->cur ^= 1;
        c->state = ST_NATURAL;
    }
    if (rc == LBM_OK && last) rc = launch_kind(c, K_FORCE, c->params(nullptr, nullptr), false);
    return rc;
}

int sync(lbm_ctx* c, const char* what) {
    LBM_CUDA(cudaMemcpyAsync(c->fault_host, c->fault_dev, sizeof(int), cudaMemcpyDeviceToHost,
                             c->stream), what);
    LBM_CUDA(cudaStreamSynchronize(c->stream), what);
    if (*c->fault_host)
        return fail(LBM_ETIMEOUT, "%s: a staged-gather kernel gave up waiting for its copies (code %d); "
                    "the state is not valid", what, *c->fault_host);
    return LBM_OK;
}

// INLET cells are producers in the step kernels: their post-collision slots carry the reservoir's
// f_eq(rho_in, u_in) where the next step's pulls read them.  A change of the flags or of the inlet
// state while the buffer holds a post-collision state rewrites those slots (enqueued on the
// context stream); a natural state needs nothing (the next step's kernels write them).
int refill_inlets(lbm_ctx* c, const char* what) {
    if (!c->any_inlet || (c->state != ST_POST_AA && c->state != ST_POST_AB)) return LBM_OK;
    void* buf = c->state_buffer();
    LBM_CUDA(c->ops->fill_inlet(c->params(buf, buf), c->state, c->grid, c->block, c->stream), what);
    ++c->launches;
    return LBM_OK;
}

// Steps per graph: even, so a chunk returns the AA parity and the A-B buffer index to where it
// started and one captured graph serves every chunk of a long run.
constexpr int kGraphChunk = 32;

// Capture `len` steps (the last one with the force when `force`) from the context's current
// state into an executable graph.  The context's state is left as it was.
int capture_steps(lbm_ctx* c, int len, bool force, lbm_ctx::GraphEntry* out) {
    if (!c->capture_stream)
        LBM_CUDA(cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking),
                 "lbm_step: capture stream");
    const int state = c->state, cur = c->cur;
    const size_t triples = c->force_triples;
    const int64_t launches = c->launches;
    cudaStream_t user = c->stream;
    c->stream = c->capture_stream;
    cudaGraph_t graph = nullptr;
    int rc = LBM_OK;
    cudaError_t e = cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        for (int i = 0; i < len && rc == LBM_OK; ++i) rc = step_once(c, force && i == len - 1);
        cudaError_t e2 = cudaStreamEndCapture(c->stream, &graph);
        if (rc == LBM_OK && e2 != cudaSuccess) rc = cuda_fail(e2, "lbm_step: end capture");
    } else {
        rc = cuda_fail(e, "lbm_step: begin capture");
    }
    c->stream = user;
    out->len = len;
    out->state = state;
    out->cur = cur;
    out->force = force;
    out->kernels = c->launches - launches;
    const size_t force_triples = c->force_triples;
    c->state = state;
    c->cur = cur;
    c->force_triples = force ? force_triples : triples;
    c->launches = launches;
    if (rc == LBM_OK) {
        e = cudaGraphInstantiate(&out->exec, graph, 0);
        if (e != cudaSuccess) rc = cuda_fail(e, "lbm_step: instantiate");
    }
    if (graph) cudaGraphDestroy(graph);
    return rc;
}

// Replays `len` steps through a cached graph (captured on first use), then advances the state
// the way the steps do.
int graph_steps(lbm_ctx* c, int len, bool force) {
    lbm_ctx::GraphEntry* g = nullptr;
    for (auto& ge : c->graphs)
        if (ge.len == len && ge.state == c->state && ge.cur == c->cur && ge.force == (int)force)
            g = &ge;
    if (!g) {
        lbm_ctx::GraphEntry ne{};
        if (int rc = capture_steps(c, len, force, &ne)) return rc;
        c->graphs.push_back(ne);
        g = &c->graphs.back();
    }
    LBM_CUDA(cudaGraphLaunch(g->exec, c->stream), "lbm_step: graph launch");
    c->launches += g->kernels;
    // state after `len` steps
    if (c->streaming == LBM_STREAMING_AA) {
        if (len & 1) c->state = c->state == ST_NATURAL ? ST_POST_AA : ST_NATURAL;
    } else {
        if (len & 1) c->cur ^= 1;
        if (c->streaming == LBM_STREAMING_AB) c->state = ST_POST_AB;
    }
    return LBM_OK;
}

}  // namespace

extern "C" {

// every call that reads or changes the state, the buffers, the stream or the launch geometry
// waits until an open slab step is ended
static int split_open(const char* what) {
    return fail(LBM_ESTATE, "%s: a slab step is open (lbm_slab_step_begin without lbm_slab_step_end)",
                what);
}

const char* lbm_last_error(void) { return g_err.c_str(); }

lbm_ctx* lbm_create(int nx, int ny, int nz, float tau, int layout, int streaming) {
    g_err.clear();
    if (nx < 1 || ny < 1 || nz < 1) {
        fail(LBM_EINVAL, "lbm_create: grid %d x %d x %d: every extent must be >= 1", nx, ny, nz);
        return nullptr;
    }
    if (ny > 65535 || nz > 65535) {
        fail(LBM_EINVAL, "lbm_create: ny and nz must be <= 65535 (got %d, %d)", ny, nz);
        return nullptr;
    }
    const size_t N = (size_t)nx * (size_t)ny * (size_t)nz;
    if (N > 2147483647u) {
        fail(LBM_EINVAL, "lbm_create: %zu cells exceed the limit of 2^31 - 1", N);
        return nullptr;
    }
    if (!std::isfinite(tau) || !(tau > 0.5f)) {
        fail(LBM_EINVAL, "lbm_create: tau = %g: need a finite tau > 1/2 (omega = 1/tau < 2)",
             (double)tau);
        return nullptr;
    }
    const LayoutOps* ops = ops_for(layout);
    if (!ops) {
        fail(LBM_EINVAL, "lbm_create: unknown layout %d", layout);
        return nullptr;
    }
    if (streaming < LBM_STREAMING_AUTO || streaming > LBM_STREAMING_AB2) {
        fail(LBM_EINVAL, "lbm_create: unknown streaming scheme %d", streaming);
        return nullptr;
    }
    if (std::getenv("LBM_FAIL_ALLOC")) {
        fail(LBM_ENOMEM, "lbm_create: allocation refused (LBM_FAIL_ALLOC is set)");
        return nullptr;
    }
    lbm_ctx* c = new (std::nothrow) lbm_ctx();
    if (!c) {
        fail(LBM_ENOMEM, "lbm_create: host allocation failed");
        return nullptr;
    }
    c->n[0] = nx;
    c->n[1] = ny;
    c->n[2] = nz;
    c->N = N;
    c->tau = tau;
    c->omega = 1.0f / tau;
    c->layout = layout;
    c->streaming = streaming == LBM_STREAMING_AUTO ? LBM_STREAMING_AA : streaming;
    c->ops = ops;
    const double u0[3] = {0.0, 0.0, 0.0};
    shifted_equilibrium(1.0, u0, c->heq_in);
    unsigned bx = 32;
    while (bx < (unsigned)nx && bx < 256) bx *= 2;
    c->block = dim3(bx, 256 / bx, 1);
    c->grid = dim3((unsigned)((nx + bx - 1) / bx), (unsigned)((ny + c->block.y - 1) / c->block.y),
                   (unsigned)nz);
    c->nblocks = (size_t)c->grid.x * c->grid.y * c->grid.z;
    const unsigned npairs = (unsigned)((nx + 1) / 2);
    unsigned bp = 32;
    while (bp < npairs && bp < 256) bp *= 2;
    c->block2 = dim3(bp, 256 / bp, 1);
    c->grid2 = dim3((npairs + bp - 1) / bp, (unsigned)((ny + c->block2.y - 1) / c->block2.y),
                    (unsigned)nz);
    c->nblocks2 = (size_t)c->grid2.x * c->grid2.y * c->grid2.z;
    if (nx % 16 == 0 && nx <= 512) {
        // persistent grid of the TMA-staged odd kernel: one CTA per SM, at most one per tile
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
            const long long tiles = ((long long)ny * nz + (512 / nx) - 1) / (512 / nx);
            c->ntma = (unsigned)std::min<long long>(sms, tiles);
        } else {
            cudaGetLastError();
        }
    }
    if (layout == LBM_LAYOUT_COLLISION && nx % kTileX == 0) {
        // tiles of 32 x 8 cells; the z planes split into chunks.  A block's time grows with the
        // planes it loads (its chunk and two halo planes) and the grid runs in waves of 2 resident
        // blocks per SM, so the count minimises waves x (chunk + 2), over chunks of at least 4
        // planes, preferring grids of at least one full wave.  Measured against about 16 blocks
        // per SM in chunks of at least 8 planes: collision AA odd step 128^3 0.142 -> 0.123 ms,
        // 256^3 0.843 -> 0.815 ms; A-B pull 0.082 -> 0.073 ms and 0.475 -> 0.454 ms.
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0) {
            const long long tiles = (long long)(nx / kTileX) * ((ny + kTileY - 1) / kTileY);
            const long long slots = 2LL * sms;
            long long chunks = 1, best = -1;
            bool best_full = false;
            for (long long ch = 1; ch <= nz; ++ch) {
                const long long len = (nz + ch - 1) / ch;
                if ((ch - 1) * len >= nz) continue;  // the last chunk would be empty
                if (len < 4 && ch > 1) break;
                const long long blocks = tiles * ch;
                const bool full = blocks >= slots;
                const long long cost = ((blocks + slots - 1) / slots) * (len + 2);
                if (best < 0 || (full && !best_full) || (full == best_full && cost < best)) {
                    best = cost;
                    best_full = full;
                    chunks = ch;
                }
            }
            c->tile_grid = dim3((unsigned)(nx / kTileX), (unsigned)((ny + kTileY - 1) / kTileY),
                                (unsigned)chunks);
            c->ntile = (size_t)c->tile_grid.x * c->tile_grid.y * c->tile_grid.z;
            // its shared memory (97 KB) is above the default limit: raised here, before any
            // stream capture; without it the pull stays element-wise
            if (c->ops->tile_prepare() != cudaSuccess) {
                cudaGetLastError();
                c->ntile = 0;
            }
        } else {
            cudaGetLastError();
        }
    }

    auto bad = [&](cudaError_t e, const char* what) {
        cuda_fail(e, what);
        c->free_all();
        delete c;
        return nullptr;
    };
    cudaError_t e;
    const size_t pop_bytes = 19 * N * c->elem_bytes_of();
    if ((e = cudaMalloc(&c->buf[0], pop_bytes)) != cudaSuccess) return bad(e, "lbm_create: population buffer");
    if (c->streaming != LBM_STREAMING_AA &&
        (e = cudaMalloc(&c->buf[1], pop_bytes)) != cudaSuccess)
        return bad(e, "lbm_create: second population buffer");
    if ((e = cudaMalloc(&c->types, N)) != cudaSuccess) return bad(e, "lbm_create: cell types");
    if ((e = cudaMalloc(&c->flags, N)) != cudaSuccess) return bad(e, "lbm_create: cell flags");
    if ((e = cudaMalloc(&c->mask, N * sizeof(uint32_t))) != cudaSuccess) return bad(e, "lbm_create: link masks");
    if ((e = cudaMalloc(&c->count_dev, 4 * sizeof(uint32_t))) != cudaSuccess) return bad(e, "lbm_create: counter");
    if ((e = cudaMalloc(&c->stage, 3 * kForceStage * sizeof(double))) != cudaSuccess)
        return bad(e, "lbm_create: force stage");
    if ((e = cudaMalloc(&c->force_dev, 3 * sizeof(double))) != cudaSuccess) return bad(e, "lbm_create: force");
    if ((e = cudaMalloc(&c->err_dev, sizeof(int))) != cudaSuccess) return bad(e, "lbm_create: error word");
    if ((e = cudaMallocHost(&c->force_host, 3 * sizeof(double))) != cudaSuccess) return bad(e, "lbm_create: pinned force");
    if ((e = cudaMallocHost(&c->err_host, sizeof(int))) != cudaSuccess) return bad(e, "lbm_create: pinned error word");
    if ((e = cudaMalloc(&c->fault_dev, sizeof(int))) != cudaSuccess) return bad(e, "lbm_create: fault word");
    if ((e = cudaMallocHost(&c->fault_host, sizeof(int))) != cudaSuccess) return bad(e, "lbm_create: pinned fault word");
    *c->fault_host = 0;
    int prio_least = 0, prio_greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest)) != cudaSuccess)
        return bad(e, "lbm_create: stream priorities");
    if ((e = cudaStreamCreateWithPriority(&c->side_stream, cudaStreamNonBlocking, prio_greatest)) != cudaSuccess)
        return bad(e, "lbm_create: boundary stream");
    if ((e = cudaEventCreateWithFlags(&c->side_fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->side_join, cudaEventDisableTiming)) != cudaSuccess)
        return bad(e, "lbm_create: boundary stream events");
    if (const char* v = std::getenv("LBM_TEST_STAGE_TIMEOUT"); v && std::strcmp(v, "1") == 0)
        c->extra_tx = 16;
    // LBM_PROFILE=1: per-kernel event timing from the start, as lbm_profile_enable(ctx, 1)
    if (const char* v = std::getenv("LBM_PROFILE"); v && std::strcmp(v, "1") == 0)
        c->profiling = true;
    // rest state: h = f - w = 0 everywhere; all cells FLUID
    if ((e = cudaMemsetAsync(c->buf[0], 0, pop_bytes, c->stream)) != cudaSuccess) return bad(e, "lbm_create: init");
    if (c->buf[1] && (e = cudaMemsetAsync(c->buf[1], 0, pop_bytes, c->stream)) != cudaSuccess)
        return bad(e, "lbm_create: init");
    if ((e = cudaMemsetAsync(c->types, 0, N, c->stream)) != cudaSuccess) return bad(e, "lbm_create: init");
    if ((e = cudaMemsetAsync(c->fault_dev, 0, sizeof(int), c->stream)) != cudaSuccess) return bad(e, "lbm_create: init");
    if (classify(c) != LBM_OK) {
        c->free_all();
        delete c;
        return nullptr;
    }
    if ((e = cudaStreamSynchronize(c->stream)) != cudaSuccess) return bad(e, "lbm_create: init");
    return c;
}

int lbm_set_stream(lbm_ctx* c, void* cuda_stream) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_stream: NULL context");
    if (c->split) return split_open("lbm_set_stream");
    if (int rc = sync(c, "lbm_set_stream")) return rc;
    c->stream = (cudaStream_t)cuda_stream;
    return LBM_OK;
}

int lbm_set_flags(lbm_ctx* c, const uint8_t* flags) {
    if (!c || !flags) return fail(LBM_EINVAL, "lbm_set_flags: NULL argument");
    if (c->split) return split_open("lbm_set_flags");
    uint8_t* tmp = nullptr;
    LBM_CUDA(cudaMalloc(&tmp, c->N), "lbm_set_flags: temporary");
    int rc = LBM_OK;
    cudaError_t e = cudaMemcpyAsync(tmp, flags, c->N, cudaMemcpyDefault, c->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->err_dev, 0, sizeof(int), c->stream);
    if (e == cudaSuccess) e = launch_validate_types(tmp, c->N, c->err_dev, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->err_host, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        rc = cuda_fail(e, "lbm_set_flags");
    } else if (*c->err_host) {
        rc = fail(LBM_EINVAL, "lbm_set_flags: flag values must be 0 (FLUID), 1 (SOLID), 2 (INLET) "
                              "or 3 (MOVING_WALL)");
    } else {
        ++c->launches;
        c->drop_graphs();
        e = cudaMemcpyAsync(c->types, tmp, c->N, cudaMemcpyDeviceToDevice, c->stream);
        if (e != cudaSuccess) rc = cuda_fail(e, "lbm_set_flags");
        if (rc == LBM_OK) rc = classify(c);
        if (rc == LBM_OK) rc = refill_inlets(c, "lbm_set_flags");
        if (rc == LBM_OK) rc = sync(c, "lbm_set_flags");
    }
    cudaFree(tmp);
    return rc;
}

int lbm_set_faces(lbm_ctx* c, int fx, int fy, int fz) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_faces: NULL context");
    if (c->split) return split_open("lbm_set_faces");
    if (c->ghost && fz != LBM_PERIODIC)
        return fail(LBM_EINVAL, "lbm_set_faces: a context with ghost planes keeps its z faces PERIODIC");
    const int f[3] = {fx, fy, fz};
    for (int a = 0; a < 3; ++a) {
        if (f[a] != LBM_PERIODIC && f[a] != LBM_OPEN)
            return fail(LBM_EINVAL, "lbm_set_faces: face type %d on axis %d", f[a], a);
        if (f[a] == LBM_OPEN && c->n[a] < 2)
            return fail(LBM_EINVAL, "lbm_set_faces: an OPEN axis needs >= 2 cells (axis %d)", a);
    }
    // scratch for the AA odd step's open-face pre-gather: 19 values per face cell and side
    size_t area[3] = {(size_t)c->n[1] * c->n[2], (size_t)c->n[0] * c->n[2], (size_t)c->n[0] * c->n[1]};
    size_t total = 0, base[3][2] = {};
    for (int a = 0; a < 3; ++a)
        for (int s = 0; s < 2; ++s) {
            base[a][s] = total;
            if (f[a] == LBM_OPEN) total += 19 * area[a];
        }
    float* scratch = nullptr;
    if (total > 0 && c->streaming == LBM_STREAMING_AA)
        LBM_CUDA(cudaMalloc(&scratch, total * sizeof(float)), "lbm_set_faces: open-face scratch");
    if (int rc = sync(c, "lbm_set_faces")) {
        cudaFree(scratch);
        return rc;
    }
    c->drop_graphs();
    cudaFree(c->scratch);
    c->scratch = scratch;
    for (int a = 0; a < 3; ++a) {
        c->face[a] = f[a];
        for (int s = 0; s < 2; ++s) c->face_base[a][s] = base[a][s];
    }
    if (int rc = classify(c)) return rc;
    return sync(c, "lbm_set_faces");
}

int lbm_set_inlet(lbm_ctx* c, float rho, float ux, float uy, float uz) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_inlet: NULL context");
    if (c->split) return split_open("lbm_set_inlet");
    if (!std::isfinite(rho) || !(rho > 0.f) || !std::isfinite(ux) || !std::isfinite(uy) ||
        !std::isfinite(uz))
        return fail(LBM_EINVAL, "lbm_set_inlet: need finite rho > 0 and finite u");
    c->drop_graphs();
    c->inlet[0] = rho;
    c->inlet[1] = ux;
    c->inlet[2] = uy;
    c->inlet[3] = uz;
    const double u[3] = {ux, uy, uz};
    shifted_equilibrium(rho, u, c->heq_in);
    return refill_inlets(c, "lbm_set_inlet");
}

int lbm_set_wall_velocity(lbm_ctx* c, float ux, float uy, float uz) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_wall_velocity: NULL context");
    if (c->split) return split_open("lbm_set_wall_velocity");
    if (!std::isfinite(ux) || !std::isfinite(uy) || !std::isfinite(uz))
        return fail(LBM_EINVAL, "lbm_set_wall_velocity: u_w must be finite");
    c->drop_graphs();
    c->uw[0] = ux;
    c->uw[1] = uy;
    c->uw[2] = uz;
    return LBM_OK;
}

int lbm_set_body_force(lbm_ctx* c, float gx, float gy, float gz) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_body_force: NULL context");
    if (c->split) return split_open("lbm_set_body_force");
    if (!std::isfinite(gx) || !std::isfinite(gy) || !std::isfinite(gz))
        return fail(LBM_EINVAL, "lbm_set_body_force: g must be finite");
    c->drop_graphs();
    c->g[0] = gx;
    c->g[1] = gy;
    c->g[2] = gz;
    return LBM_OK;
}

static void reset_state(lbm_ctx* c) {
    c->state = ST_NATURAL;
    c->steps = 0;
    c->force_valid = false;
}

int lbm_set_populations(lbm_ctx* c, const float* f) {
    if (!c || !f) return fail(LBM_EINVAL, "lbm_set_populations: NULL argument");
    if (c->split) return split_open("lbm_set_populations");
    void* dst = c->state_buffer();
    const Params p = c->params(dst, dst);
    const size_t total = 19 * c->N;
    if (is_device_pointer(f)) {
        LBM_CUDA(c->ops->pack(p, f, 0, total, c->stream), "lbm_set_populations: pack");
        ++c->launches;
    } else {
        if (int rc = ensure_staging(c)) return rc;
        int k = 0;
        for (size_t i0 = 0; i0 < total; i0 += kStageHalf, ++k) {
            const size_t cnt = total - i0 < kStageHalf ? total - i0 : kStageHalf;
            const int h = k & 1;
            float* s = c->staging + h * kStageHalf;
            if (int rc = stage_in(c, h, s, f + i0, cnt)) return rc;
            if (int rc = stage_in_done(c, h)) return rc;
            LBM_CUDA(c->ops->pack(p, s, i0, cnt, c->stream), "lbm_set_populations: pack");
            ++c->launches;
            if (int rc = stage_used(c, h)) return rc;
        }
        if (int rc = stage_end(c)) return rc;
    }
    reset_state(c);
    return sync(c, "lbm_set_populations");
}

int lbm_set_equilibrium(lbm_ctx* c, const float* rho, const float* u) {
    if (!c || !rho || !u) return fail(LBM_EINVAL, "lbm_set_equilibrium: NULL argument");
    if (c->split) return split_open("lbm_set_equilibrium");
    void* dst = c->state_buffer();
    const Params p = c->params(dst, dst);
    const size_t N = c->N;
    if (is_device_pointer(rho) && is_device_pointer(u)) {
        LBM_CUDA(c->ops->equilibrium(p, rho, u, u + N, u + 2 * N, 0, (uint32_t)N, c->stream),
                 "lbm_set_equilibrium");
        ++c->launches;
    } else {
        if (int rc = ensure_staging(c)) return rc;
        const size_t chunk = kStageHalf / 4;
        int k = 0;
        for (size_t n0 = 0; n0 < N; n0 += chunk, ++k) {
            const size_t cnt = N - n0 < chunk ? N - n0 : chunk;
            const int h = k & 1;
            float* s = c->staging + h * kStageHalf;
            if (int rc = stage_in(c, h, s, rho + n0, cnt)) return rc;
            for (int a = 0; a < 3; ++a)
                LBM_CUDA(cudaMemcpyAsync(s + (a + 1) * chunk, u + a * N + n0, cnt * 4, cudaMemcpyDefault,
                                         c->copy_stream), "lbm_set_equilibrium: copy");
            if (int rc = stage_in_done(c, h)) return rc;
            LBM_CUDA(c->ops->equilibrium(p, s, s + chunk, s + 2 * chunk, s + 3 * chunk, (uint32_t)n0,
                                         (uint32_t)cnt, c->stream), "lbm_set_equilibrium");
            ++c->launches;
            if (int rc = stage_used(c, h)) return rc;
        }
        if (int rc = stage_end(c)) return rc;
    }
    reset_state(c);
    return sync(c, "lbm_set_equilibrium");
}

int lbm_get_populations(lbm_ctx* c, float* f) {
    if (!c || !f) return fail(LBM_EINVAL, "lbm_get_populations: NULL argument");
    if (c->split) return split_open("lbm_get_populations");
    void* src = c->state_buffer();
    const Params p = c->params(src, src);
    const size_t total = 19 * c->N;
    if (is_device_pointer(f)) {
        LBM_CUDA(c->ops->unpack(p, c->state, f, 0, total, c->stream), "lbm_get_populations");
        ++c->launches;
    } else {
        if (int rc = ensure_staging(c)) return rc;
        int k = 0;
        for (size_t i0 = 0; i0 < total; i0 += kStageHalf, ++k) {
            const size_t cnt = total - i0 < kStageHalf ? total - i0 : kStageHalf;
            const int h = k & 1;
            float* s = c->staging + h * kStageHalf;
            if (int rc = stage_out_begin(c, h)) return rc;
            LBM_CUDA(c->ops->unpack(p, c->state, s, i0, cnt, c->stream), "lbm_get_populations");
            ++c->launches;
            if (int rc = stage_out_ready(c, h)) return rc;
            if (int rc = stage_out(c, h, f + i0, s, cnt)) return rc;
            if (int rc = stage_out_copied(c, h)) return rc;
        }
        if (int rc = stage_end(c)) return rc;
    }
    return sync(c, "lbm_get_populations");
}

int lbm_step(lbm_ctx* c, int n) {
    if (!c) return fail(LBM_EINVAL, "lbm_step: NULL context");
    if (c->split) return split_open("lbm_step");
    if (n < 0) return fail(LBM_EINVAL, "lbm_step: n = %d < 0", n);
    if (c->ghost && n > 1)
        return fail(LBM_EINVAL, "lbm_step: with ghost planes, step once and exchange the halos "
                                "between steps (n = %d)", n);
    if (c->use_graphs && !c->profiling) {
        for (int done = 0; done < n;) {
            const int len = n - done > kGraphChunk ? kGraphChunk : n - done;
            if (int rc = graph_steps(c, len, done + len == n)) return rc;
            done += len;
        }
    } else {
        for (int i = 0; i < n; ++i)
            if (int rc = step_once(c, i == n - 1)) return rc;
    }
    if (n > 0) {
        c->steps += n;
        c->force_valid = true;
    }
    return LBM_OK;
}

int lbm_macroscopic(lbm_ctx* c, float* rho, float* u) {
    if (!c || !rho || !u) return fail(LBM_EINVAL, "lbm_macroscopic: NULL argument");
    if (c->split) return split_open("lbm_macroscopic");
    void* src = c->state_buffer();
    const Params p = c->params(src, src);
    const size_t N = c->N;
    if (is_device_pointer(rho) && is_device_pointer(u)) {
        LBM_CUDA(c->ops->macro(p, c->state, c->inlet, rho, u, u + N, u + 2 * N, 0, (uint32_t)N,
                               c->stream), "lbm_macroscopic");
        ++c->launches;
    } else {
        if (int rc = ensure_staging(c)) return rc;
        const size_t chunk = kStageHalf / 4;
        int k = 0;
        for (size_t n0 = 0; n0 < N; n0 += chunk, ++k) {
            const size_t cnt = N - n0 < chunk ? N - n0 : chunk;
            const int h = k & 1;
            float* s = c->staging + h * kStageHalf;
            if (int rc = stage_out_begin(c, h)) return rc;
            LBM_CUDA(c->ops->macro(p, c->state, c->inlet, s, s + chunk, s + 2 * chunk, s + 3 * chunk,
                                   (uint32_t)n0, (uint32_t)cnt, c->stream), "lbm_macroscopic");
            ++c->launches;
            if (int rc = stage_out_ready(c, h)) return rc;
            if (int rc = stage_out(c, h, rho + n0, s, cnt)) return rc;
            for (int a = 0; a < 3; ++a)
                if (int rc = stage_out(c, h, u + a * N + n0, s + (a + 1) * chunk, cnt)) return rc;
            if (int rc = stage_out_copied(c, h)) return rc;
        }
        if (int rc = stage_end(c)) return rc;
    }
    return sync(c, "lbm_macroscopic");
}

int lbm_force_momentum_exchange(lbm_ctx* c, double F[3]) {
    if (!c || !F) return fail(LBM_EINVAL, "lbm_force_momentum_exchange: NULL argument");
    if (c->split) return split_open("lbm_force_momentum_exchange");
    if (!c->force_valid)
        return fail(LBM_ESTATE, "lbm_force_momentum_exchange: no step since the state was loaded");
    LBM_CUDA(cudaMemcpyAsync(c->force_host, c->force_dev, 3 * sizeof(double), cudaMemcpyDeviceToHost,
                             c->stream), "lbm_force_momentum_exchange");
    if (int rc = sync(c, "lbm_force_momentum_exchange")) return rc;
    for (int a = 0; a < 3; ++a) F[a] = c->force_host[a];
    return LBM_OK;
}

int lbm_check_finite(lbm_ctx* c) {
    if (!c) return fail(LBM_EINVAL, "lbm_check_finite: NULL context");
    if (c->split) return split_open("lbm_check_finite");
    void* src = c->state_buffer();
    LBM_CUDA(cudaMemsetAsync(c->err_dev, 0, sizeof(int), c->stream), "lbm_check_finite");
    LBM_CUDA(c->ops->check_finite(c->params(src, src), c->err_dev, c->grid, c->block, c->stream),
             "lbm_check_finite");
    ++c->launches;
    LBM_CUDA(cudaMemcpyAsync(c->err_host, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost, c->stream),
             "lbm_check_finite");
    if (int rc = sync(c, "lbm_check_finite")) return rc;
    if (*c->err_host) return fail(LBM_ENOTFINITE, "lbm_check_finite: a population is NaN or infinite");
    return LBM_OK;
}

int64_t lbm_step_count(lbm_ctx* c) { return c ? c->steps : -1; }

int64_t lbm_kernel_launches(lbm_ctx* c) { return c ? c->launches : -1; }

int lbm_set_ghost_planes(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_ghost_planes: NULL context");
    if (c->split) return split_open("lbm_set_ghost_planes");
    if (enable) {
        if (c->streaming != LBM_STREAMING_AB)
            return fail(LBM_EINVAL, "lbm_set_ghost_planes: needs the A-B scheme (LBM_STREAMING_AB)");
        if (c->face[2] != LBM_PERIODIC)
            return fail(LBM_EINVAL, "lbm_set_ghost_planes: the z faces must be PERIODIC");
        if (c->n[2] < 3) return fail(LBM_EINVAL, "lbm_set_ghost_planes: needs nz >= 3");
    }
    const bool old = c->ghost;
    c->ghost = enable != 0;
    c->drop_graphs();
    const int rc = classify(c);
    if (rc != LBM_OK) c->ghost = old;
    return rc;
}

int64_t lbm_halo_elements(lbm_ctx* c) {
    return c ? 5 * (int64_t)c->n[0] * (int64_t)c->n[1] : -1;
}

int lbm_halo_element_bytes(lbm_ctx* c) {
    if (!c) return fail(LBM_EINVAL, "lbm_halo_element_bytes: NULL context");
    return (int)c->elem_bytes_of();
}

// Halo buffers are device memory of the context's device (they go to a communication library).
static int check_halo_buffers(lbm_ctx* c, const void* a, const void* b, const char* what) {
    if (!c || !a || !b) return fail(LBM_EINVAL, "%s: NULL argument", what);
    if (!c->ghost) return fail(LBM_ESTATE, "%s: the context has no ghost planes", what);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(LBM_ECUDA, "%s: no current device", what);
    }
    for (const void* ptr : {a, b}) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
            cudaGetLastError();
            return fail(LBM_EINVAL, "%s: halo buffers must be device memory", what);
        }
        if (!(at.type == cudaMemoryTypeManaged || (at.type == cudaMemoryTypeDevice && at.device == dev)))
            return fail(LBM_EINVAL, "%s: halo buffers must be device memory of the current device", what);
    }
    return LBM_OK;
}
static int check_halo(lbm_ctx* c, const void* a, const void* b, const char* what) {
    if (int rc = check_halo_buffers(c, a, b, what)) return rc;
    if (c->state != ST_POST_AB)
        return fail(LBM_ESTATE, "%s: no step taken since the state was loaded", what);
    return LBM_OK;
}

int lbm_halo_pack(lbm_ctx* c, void* lo, void* hi) {
    if (c && c->split) return split_open("lbm_halo_pack");
    if (int rc = check_halo(c, lo, hi, "lbm_halo_pack")) return rc;
    void* buf = c->buf[c->cur];
    LBM_CUDA(c->ops->halo_pack(c->params(buf, buf), lo, hi, c->stream), "lbm_halo_pack");
    ++c->launches;
    return LBM_OK;
}

int lbm_halo_unpack(lbm_ctx* c, const void* from_below, const void* from_above) {
    if (c && c->split) return split_open("lbm_halo_unpack");
    if (int rc = check_halo(c, from_below, from_above, "lbm_halo_unpack")) return rc;
    void* buf = c->buf[c->cur];
    LBM_CUDA(c->ops->halo_unpack(c->params(buf, buf), from_below, from_above, c->stream),
             "lbm_halo_unpack");
    ++c->launches;
    return LBM_OK;
}

// ---- slab step with the halo exchange overlapped ------------------------------------------------
// The main kernel of step kind `kind` over `count` planes z = z0 + dz k (k < count), then the
// boundary kernel over special[s0, s1), both on stream `s`, with the momentum exchange; their
// force partials take the triples from `slot` on (advanced past them).
static int launch_planes(lbm_ctx* c, int kind, const Params& p0, int z0, int dz, int count,
                         uint32_t s0, uint32_t s1, size_t& slot, cudaStream_t s) {
    if (count > 0) {
        Params p = p0;
        p.zbase = z0;
        p.zstep = dz;
        p.part_main = slot;
        const bool two = c->pairs_for(kind);
        dim3 grid = two ? c->grid2 : c->grid;
        grid.z = (unsigned)count;
        const cudaError_t e = two ? c->ops->cells2(kind, p, true, c->body(), grid, c->block2, s)
                                  : c->ops->cells(kind, p, true, c->body(), grid, c->block, s);
        ++c->launches;
        if (e != cudaSuccess) return cuda_fail(e, "slab step: kernel launch");
        slot += (size_t)grid.x * grid.y * grid.z * kWarpsPerBlock;
    }
    if (kind == K_AB_PULL && s1 > s0) {
        Params p = p0;
        p.special = c->special + s0;
        p.n_special = s1 - s0;
        p.part_special = slot;
        const cudaError_t e = c->ops->special(K_AB_PULL, p, true, c->body(), s);
        ++c->launches;
        if (e != cudaSuccess) return cuda_fail(e, "slab step: boundary kernel launch");
        slot += (size_t)special_blocks(s1 - s0) * kWarpsPerBlock;
    }
    return LBM_OK;
}

// Force partial triples of a slab step (the launches of lbm_slab_step_begin): the main kernel over
// the owned planes 1 .. nz - 2, and for the pull the boundary kernel over the special cells, split
// at the edge planes into `edges` + 1 ranges (one range for a slab that owns one plane).
static size_t slab_step_triples(const lbm_ctx* c, int kind, int edges) {
    const bool two = c->pairs_for(kind);
    const dim3 g = two ? c->grid2 : c->grid;
    size_t blocks = (size_t)g.x * g.y * (size_t)(c->n[2] - 2);
    if (kind == K_AB_PULL) {
        if (edges == 2)
            blocks += special_blocks(c->sp_lo_end) + special_blocks(c->n_special - c->sp_hi_begin) +
                      special_blocks(c->sp_hi_begin - c->sp_lo_end);
        else
            blocks += special_blocks(c->n_special);
    }
    return blocks * kWarpsPerBlock;
}

int lbm_slab_step_begin(lbm_ctx* c, void* lo, void* hi) {
    if (c && c->split)
        return fail(LBM_ESTATE, "lbm_slab_step_begin: the previous slab step is still open");
    if (int rc = check_halo_buffers(c, lo, hi, "lbm_slab_step_begin")) return rc;
    const int nz = c->n[2];
    // a step from the loaded (natural) state is the collision alone, as in lbm_step
    const int kind = c->state == ST_NATURAL ? K_AB_COLLIDE : K_AB_PULL;
    void* dst = c->buf[c->cur ^ 1];
    const Params p = c->params(c->buf[c->cur], dst);
    // the edge planes 1 and nz - 2 (one plane when the slab owns one), their special cells, and
    // the pack of their outgoing populations, on the context stream
    const int edges = nz - 2 > 1 ? 2 : 1;
    // the kernels' force partials must fit before any of them is launched
    const size_t need = slab_step_triples(c, kind, edges);
    if (need > c->partial_cap)
        return fail(LBM_ESTATE, "lbm_slab_step_begin: %zu force partials exceed the %zu allocated",
                    need, c->partial_cap);
    size_t slot = 0;
    int rc = launch_planes(c, kind, p, 1, nz - 3, edges, 0, 0, slot, c->stream);
    if (rc == LBM_OK) {
        if (edges == 2) {
            rc = launch_planes(c, kind, p, 0, 0, 0, 0, c->sp_lo_end, slot, c->stream);
            if (rc == LBM_OK)
                rc = launch_planes(c, kind, p, 0, 0, 0, c->sp_hi_begin, c->n_special, slot, c->stream);
        } else {
            rc = launch_planes(c, kind, p, 0, 0, 0, 0, c->n_special, slot, c->stream);
        }
    }
    if (rc != LBM_OK) return rc;
    LBM_CUDA(c->ops->halo_pack(c->params(dst, dst), lo, hi, c->stream), "lbm_slab_step_begin: pack");
    ++c->launches;
    // the interior planes 2 .. nz - 3 and their special cells on the side stream, forked after the
    // pack: a transfer the caller orders after the context stream's work so far runs beside them
    LBM_CUDA(cudaEventRecord(c->side_fork, c->stream), "lbm_slab_step_begin: fork");
    LBM_CUDA(cudaStreamWaitEvent(c->side_stream, c->side_fork, 0), "lbm_slab_step_begin: fork");
    if (edges == 2)
        rc = launch_planes(c, kind, p, 2, 1, nz - 4, c->sp_lo_end, c->sp_hi_begin, slot, c->side_stream);
    cudaError_t e = cudaEventRecord(c->side_join, c->side_stream);
    if (rc != LBM_OK) {
        if (e == cudaSuccess) cudaStreamWaitEvent(c->stream, c->side_join, 0);
        return rc;
    }
    if (e != cudaSuccess) return cuda_fail(e, "lbm_slab_step_begin: join");
    c->force_triples = slot;
    c->split = true;
    return LBM_OK;
}

int lbm_slab_step_end(lbm_ctx* c, const void* from_below, const void* from_above) {
    if (c && !c->split) return fail(LBM_ESTATE, "lbm_slab_step_end: no slab step is open");
    if (int rc = check_halo_buffers(c, from_below, from_above, "lbm_slab_step_end")) return rc;
    LBM_CUDA(cudaStreamWaitEvent(c->stream, c->side_join, 0), "lbm_slab_step_end: join");
    c->split = false;
    c->cur ^= 1;
    c->state = ST_POST_AB;
    c->steps += 1;
    LBM_CUDA(launch_force_finalize(c->partial, c->force_triples, c->stage, c->force_dev, c->stream),
             "lbm_slab_step_end: force");
    c->launches += 2;
    c->force_valid = true;
    void* buf = c->buf[c->cur];
    LBM_CUDA(c->ops->halo_unpack(c->params(buf, buf), from_below, from_above, c->stream),
             "lbm_slab_step_end: unpack");
    ++c->launches;
    return LBM_OK;
}

int lbm_profile_enable(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_profile_enable: NULL context");
    if (c->split) return split_open("lbm_profile_enable");
    if (int rc = sync(c, "lbm_profile_enable")) return rc;
    c->release_profile();
    c->profiling = enable != 0;
    return LBM_OK;
}

int lbm_profile_read(lbm_ctx* c, int kind, int64_t* launches, double* total_ms) {
    if (!c || !launches || !total_ms) return fail(LBM_EINVAL, "lbm_profile_read: NULL argument");
    if (c->split) return split_open("lbm_profile_read");
    if (kind < 0 || kind >= K_NUM_KINDS) return fail(LBM_EINVAL, "lbm_profile_read: kind %d", kind);
    if (int rc = sync(c, "lbm_profile_read")) return rc;
    double ms = 0.0;
    for (auto& pr : c->prof[kind]) {
        float t = 0.f;
        LBM_CUDA(cudaEventElapsedTime(&t, pr.first, pr.second), "lbm_profile_read");
        ms += t;
    }
    *launches = (int64_t)c->prof[kind].size();
    *total_ms = ms;
    return LBM_OK;
}

int lbm_set_cell_pairs(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_cell_pairs: NULL context");
    if (c->split) return split_open("lbm_set_cell_pairs");
    if (c->pairs_allowed != (enable != 0)) {
        c->drop_graphs();
        c->pairs_allowed = enable != 0;
    }
    return c->pairs() ? 1 : 0;
}

int lbm_set_tma_gather(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_tma_gather: NULL context");
    if (c->split) return split_open("lbm_set_tma_gather");
    if (c->tma_allowed != (enable != 0)) {
        c->drop_graphs();
        c->tma_allowed = enable != 0;
    }
    return c->tma() ? 1 : 0;
}

int lbm_set_boundary_overlap(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_boundary_overlap: NULL context");
    if (c->split) return split_open("lbm_set_boundary_overlap");
    if (c->overlap_allowed != (enable != 0)) {
        c->drop_graphs();
        c->overlap_allowed = enable != 0;
    }
    return LBM_OK;
}

int lbm_set_graph_launch(lbm_ctx* c, int enable) {
    if (!c) return fail(LBM_EINVAL, "lbm_set_graph_launch: NULL context");
    if (c->split) return split_open("lbm_set_graph_launch");
    c->use_graphs = enable != 0;
    return LBM_OK;
}

void lbm_destroy(lbm_ctx* c) {
    if (!c) return;
    c->free_all();
    delete c;
}

}  // extern "C"
