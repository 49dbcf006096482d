/*
 * lbm.h -- C ABI of the GB300 D3Q19 BGK lattice Boltzmann library (liblbm.so).
 *
 * One context = one dense nx*ny*nz lattice on the current CUDA device, advanced by fused
 * stream-collide kernels on one CUDA stream.  Sources, cited by page title and section:
 *
 *  [PortLBM]  "PortLBM: A Portable Lattice Boltzmann Tool Leveraging SYCL on AMD, NVIDIA, and
 *             Intel GPUs": §3.1 Eq. 1 (BGK update, time step 1), Eq. 2 (second-order
 *             equilibrium, 2D incompressible variant), last paragraph of §3.1 (equilibrium inlet,
 *             halfway bounce-back, outlet), §3.2 and Fig. 2 (stream / collision / bundle
 *             layouts), §3.3 Eq. 3 (collision + streaming; one-step pull, two lattices).
 *  [Layout]   "GPU lattice Boltzmann: streaming layout and performance": the "In place" bullet
 *             (AA addressing, 152 population bytes per cell update), the "Two buffers" bullet
 *             (collide in place, then pull: 304 bytes), the paragraph after them (the same
 *             per-link wall / reflection / open-face rules in both; gather before scatter; the
 *             momentum exchange of a submission's last step), and `Streaming::Auto`.
 *  [Blog]     "GPU加速LBM流体仿真：从原理到150倍性能优化实战": §2.2 (D3Q19 weights 1/3, 1/18,
 *             1/36), §5.1 (omega = 1/(3 nu + 1/2): stability requires tau > 1/2).
 *
 * Velocity set (fixed by this ABI; [Blog] §2.2 gives the classes rest / 6 axis / 12 diagonal):
 *   q : 0 (0,0,0)   1 (+1,0,0)  2 (-1,0,0)  3 (0,+1,0)  4 (0,-1,0)  5 (0,0,+1)  6 (0,0,-1)
 *       7 (+1,+1,0) 8 (-1,-1,0) 9 (+1,0,+1) 10 (-1,0,-1) 11 (0,+1,+1) 12 (0,-1,-1)
 *       13 (+1,-1,0) 14 (-1,+1,0) 15 (+1,0,-1) 16 (-1,0,+1) 17 (0,+1,-1) 18 (0,-1,+1)
 *   weights w0 = 1/3, w1..w6 = 1/18, w7..w18 = 1/36; opposite(q) = q+1 for odd q, q-1 for even
 *   q > 0, opposite(0) = 0.
 *
 * Canonical array conventions at this ABI (the internal layout is never visible):
 *   cell index  n = x + nx*(y + ny*z), N = nx*ny*nz;
 *   populations f[q*N + n], fp32, absolute values, the natural (pre-collision) state f(x, t);
 *   flags       uint8 per cell: LBM_FLUID, LBM_SOLID (bounce-back), LBM_INLET (reservoir held at
 *               f_eq(rho_in, u_in), never updated), LBM_MOVING_WALL (bounce-back off a wall moving
 *               at u_w);
 *   rho[n], u[a*N + n] (a = 0,1,2), fp32.
 *
 * The step.  Per time step every FLUID cell x collides (BGK, relaxation omega = 1/tau,
 * equilibrium w rho [1 + 3 c.u + 9/2 (c.u)^2 - 3/2 u.u], c_s^2 = 1/3; with a body acceleration g
 * Guo forcing: F = rho g, u = j/rho + g/2, source (1 - omega/2) w [3 (c - u).F + 9 (c.u)(c.F)])
 * and then receives population q from s = x - c_q, wrapped on PERIODIC axes and clamped onto the
 * last layer on OPEN axes (zero-gradient): FLUID s gives its post-collision f*_q(s); SOLID s
 * reflects x's own f*_opposite(q)(x) (halfway bounce-back); INLET s gives f_eq,q(rho_in, u_in);
 * MOVING_WALL s reflects f*_opposite(q)(x) + 2 w_q (c_q.u_w)/c_s^2 ([Blog] §4.2, the mirror method,
 * at the reference density 1).
 *
 * Ownership and threading.  The caller owns every array it passes; the library keeps no caller
 * pointer after a call returns.  Array arguments may be device pointers or host pointers (pinned
 * or pageable); host data is staged through the library's own buffers.  A context is used by one
 * host thread at a time.  Calls that only enqueue work (lbm_step) are asynchronous on the
 * context's stream; calls that return data to the caller synchronise that stream.
 *
 * Changes between steps.  After an odd number of AA steps, and after any A-B step, the buffer holds
 * post-collision values whose streaming (the second half of the last step) is still pending; a
 * change of the flags, faces, inlet state or wall velocity made then acts on that streaming, as it
 * does on every later step.  After an even number of AA steps and in the AB2 scheme the state is
 * natural and a change acts from the next step on.
 *
 * Errors.  Functions returning int give LBM_OK (0) or a negative LBM_E* code; lbm_create returns
 * NULL on failure.  The message for the calling thread's last failure is lbm_last_error().  A call
 * that fails argument validation changes nothing; a CUDA failure (LBM_ECUDA) leaves the context
 * usable only for lbm_destroy.
 */
#ifndef LBM_H
#define LBM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lbm_ctx lbm_ctx;

/* Population layouts ([PortLBM] §3.2, Fig. 2).  STREAM: SoA, f[q][n].  COLLISION: AoS,
 * f[n][q].  BUNDLE: SoAoS; the populations are grouped by (c_y, c_z) into 9 bundles (the x-rows
 * of the stencil: five of three members ordered c_x = -1, 0, +1, four of one), and bundle b of
 * size m_b stores f[b-offset*N + n*m_b + j]. */
enum { LBM_LAYOUT_STREAM = 0, LBM_LAYOUT_BUNDLE = 1, LBM_LAYOUT_COLLISION = 2,
       LBM_LAYOUT_STREAM_FP16 = 3 };
/* LBM_LAYOUT_STREAM_FP16: the stream layout with the populations stored as IEEE half precision
 * (shifted by their weights, f - w; arithmetic stays fp32, one round-to-nearest per store): 76
 * population bytes per cell update instead of 152.  Each stored population keeps 11 significant
 * bits, so per-step changes below half a unit of the stored value are rounded away: a channel
 * driven by a body force of 1e-6 reaches 96% of the fp32 centre-line velocity after 2000 steps,
 * the drag of a sphere is accurate to about 1e-3 relative, a Taylor-Green vortex to 3e-6 after
 * 100 steps.  |f - w| must stay below 65504.  ([Blog] §5.2 suggests half-precision storage for
 * a bandwidth-bound step and leaves its precision loss to be checked; no page fixes a format.) */

/* Streaming schemes.  AA ([Layout] "In place"): one buffer; even steps read (q, x) and write the
 * collided value at (opposite(q), x); odd steps read (opposite(q), x - c_q) and write (q, x + c_q);
 * 152 population bytes per cell update.  AB: two buffers, fused pull-collide ([PortLBM] §3.3
 * one-step pull two-lattice), also 152 bytes per update.  AB2: two buffers, [Layout] "Two
 * buffers" form: collide in place, then pull into the other buffer, 304 bytes per update.  AUTO
 * resolves to AA, as [Layout]'s `Streaming::Auto` does. */
enum { LBM_STREAMING_AUTO = 0, LBM_STREAMING_AA = 1, LBM_STREAMING_AB = 2, LBM_STREAMING_AB2 = 3 };

enum {
    LBM_OK = 0,
    LBM_EINVAL = -1,     /* invalid argument                                               */
    LBM_ENOMEM = -2,     /* device or host allocation failed                               */
    LBM_ECUDA = -3,      /* CUDA runtime error (message in lbm_last_error)                  */
    LBM_ESTATE = -4,     /* call not valid in the current state (e.g. force before a step)  */
    LBM_ENOTFINITE = -5, /* lbm_check_finite found a NaN or infinity                         */
    LBM_ETIMEOUT = -6    /* a bounded wait inside a kernel ran out (state not valid)        */
};

enum { LBM_FLUID = 0, LBM_SOLID = 1, LBM_INLET = 2, LBM_MOVING_WALL = 3 };
enum { LBM_PERIODIC = 0, LBM_OPEN = 1 };

/* Create a context on the current CUDA device.  nx, ny, nz >= 1, nz <= 65535, N <= 2^31 - 1,
 * tau > 1/2 and finite ([Blog] §5.1: omega = 1/tau must stay below 2).  Allocates the population
 * buffer(s) (AA: one, AB/AB2: two, 76 N bytes each, 38 N in half-precision storage), the cell
 * type and flag bytes and the solid-link masks (6 N bytes).  Initial state: every cell
 * FLUID, all faces PERIODIC, g = 0, inlet (1, 0, 0, 0), f = w_q (rest at rho = 1), step count 0,
 * stream 0 (the legacy default stream).  Returns NULL on error (see lbm_last_error). */
lbm_ctx* lbm_create(int nx, int ny, int nz, float tau, int layout, int streaming);

/* Message for the calling thread's most recent failure ("" if none).  Valid until that thread's
 * next call into the library.  (No page defines an error interface; [PortLBM] §4 names only an
 * abstract handler that initialises and controls a simulation.  Status codes with a per-thread
 * message are this ABI's own convention.) */
const char* lbm_last_error(void);

/* Use `cuda_stream` (a cudaStream_t, e.g. torch.cuda.current_stream().cuda_stream) for all later
 * work of this context.  Work already enqueued on the previous stream is synchronised first.
 * ([Layout] submits a flow's steps as submissions to one device queue and reads the forces of a
 * submission's last step; the CUDA stream is that queue here.  The stream belongs to the caller
 * and must stay valid while the context uses it.) */
int lbm_set_stream(lbm_ctx* ctx, void* cuda_stream);

/* Cell flags, N bytes, LBM_FLUID / LBM_SOLID / LBM_INLET / LBM_MOVING_WALL ([PortLBM] §3.1
 * boundary treatment; [Blog] §4.2 moving walls; [Layout]: the per-link rules are driven by the
 * cell type).  Any other value -> LBM_EINVAL.
 * Changing flags does not touch the FLUID cells' populations; INLET cells, which the step kernels
 * run as producers of f_eq(rho_in, u_in), get their outgoing slots rewritten when streaming is
 * pending (see "Changes between steps" above).  Synchronous. */
int lbm_set_flags(lbm_ctx* ctx, const uint8_t* flags);

/* Face type per axis: LBM_PERIODIC (wrap) or LBM_OPEN (zero-gradient: a population whose source
 * lies beyond the face comes from the source clamped onto the last layer).  An OPEN axis needs at
 * least 2 cells; any other value -> LBM_EINVAL, nothing changed.  ([PortLBM] §3.1, last
 * paragraph: Neumann-type outlet; [Layout]: open-face rules are per-link rules.  Periodic wrap
 * is the pages' periodic 128^3 case.) */
int lbm_set_faces(lbm_ctx* ctx, int face_x, int face_y, int face_z);

/* State held by every INLET cell: f = f_eq(rho, (ux, uy, uz)).  rho > 0 and finite, u finite;
 * otherwise LBM_EINVAL, nothing changed.  The step kernels run INLET cells as producers: their
 * outgoing slots carry f_eq where a FLUID cell's post-collision values would be, so that their
 * neighbours take the ordinary path.  When streaming is pending (see "Changes between steps"
 * above) this call enqueues a small kernel on the context stream that rewrites those slots;
 * asynchronous.  ([PortLBM] §3.1, last paragraph: the inlet imposes the equilibrium
 * distribution.) */
int lbm_set_inlet(lbm_ctx* ctx, float rho, float ux, float uy, float uz);

/* Velocity u_w of every LBM_MOVING_WALL cell ([Blog] §4.2).  Finite; 0 (the initial value) makes
 * moving walls behave as solid ones. */
int lbm_set_wall_velocity(lbm_ctx* ctx, float ux, float uy, float uz);

/* Body acceleration g (force density F = rho g), applied with Guo forcing.  0 disables it; a
 * non-finite component -> LBM_EINVAL, nothing changed.  (No page describes the forcing scheme:
 * reading R4 of this library's design notes, Guo forcing with the half-force velocity shift
 * u = j/rho + g/2 and the source (1 - omega/2) w [3 (c - u).F + 9 (c.u)(c.F)].) */
int lbm_set_body_force(lbm_ctx* ctx, float gx, float gy, float gz);

/* Load the natural state f(x, t) from f[19*N] (canonical, absolute fp32).  Values of SOLID and
 * INLET cells are ignored.  Resets the step count to 0 (AA even parity).  Synchronous.
 * ([Layout] "In place": at an even step count the buffer holds population q of cell x at (q, x),
 * so loading is a layout change plus the weight shift; in the two-buffer schemes it fills the
 * source buffer.) */
int lbm_set_populations(lbm_ctx* ctx, const float* f);

/* Load f = f_eq(rho[n], u[.][n]) for every FLUID cell, computed on the device in fp32
 * ([PortLBM] Eq. 2 in its 3D compressible form).  rho[N] > 0, u[3*N].  Resets the step count to 0.
 * Synchronous. */
int lbm_set_equilibrium(lbm_ctx* ctx, const float* rho, const float* u);

/* Read the natural state f(x, t) into f[19*N] (canonical, absolute fp32), whatever the AA parity
 * or A-B buffer state: after an odd AA step count the streaming half of the next step is applied
 * on the fly.  SOLID and MOVING_WALL cells read 0, INLET cells f_eq(rho_in, u_in).
 * Synchronous.  ([Layout] "In place": after an odd step the collided population q of cell x sits
 * at (opposite(q), x) and reaches x + c_q only in the next step's read, which the decoder
 * applies through the per-link rules.) */
int lbm_get_populations(lbm_ctx* ctx, float* f);

/* Enqueue n >= 0 time steps ([PortLBM] Eq. 1 with the per-link rules above) on the context
 * stream.  The last of the n steps also computes the momentum-exchange force of its
 * post-collision state (read with lbm_force_momentum_exchange).  Asynchronous; n = 0 is a no-op
 * that leaves the last force unchanged.  With graph launch on (the default) the steps are
 * replayed from CUDA graphs of up to 32 steps, captured on a private stream on first use and
 * cached per (length, buffer state); the setters of flags, faces, inlet, wall velocity and body
 * force drop the cache.  Results are identical with graph launch on or off. */
int lbm_step(lbm_ctx* ctx, int n);

/* Turn graph replay of lbm_step on (enable != 0, the default) or off (one launch per kernel).
 * While per-kernel profiling is enabled, steps are always launched one by one. */
int lbm_set_graph_launch(lbm_ctx* ctx, int enable);

/* Allow (enable != 0, the default) or forbid the two-cell step kernels: one thread updates the
 * x-adjacent cells (x, x+1), x even, loading and storing the pair's aligned slots as one word and
 * colliding both cells in packed fp32x2 arithmetic.  They serve the stream layouts (fp32 and
 * fp16 storage) when nx is even and 19 N <= 2^32, and on those grids the bundle layout's AA even
 * step too (a pair's records of one bundle are one aligned run); elsewhere one thread updates one
 * cell.  The
 * populations are bit-identical either way; the momentum-exchange force may differ in its last
 * bits (its partial sums are grouped by thread).  Populations of non-FLUID cells are not defined
 * under either kernel family: a cell turned FLUID by lbm_set_flags needs its populations set.
 * Returns 1 when the stream layouts' two-cell kernels will run, 0 when they will not, LBM_EINVAL
 * for a NULL context.  Drops the cached step graphs.  (No page prescribes this mapping; it is a launch
 * choice for the same update.) */
int lbm_set_cell_pairs(lbm_ctx* ctx, int enable);

/* Allow (enable != 0) or forbid (enable = 0, the default) the TMA-staged AA odd step: an
 * alternative AA odd kernel, off by default because it measured slower than the register-addressed
 * two-cell kernel on every workload tried (512^3: 12.5 vs 3.1 ms).  Persistent CTAs (one per
 * SM) stage each tile's source rows -- every population plane, plus the tile's own rows, flags
 * and solid-link masks when the domain has solid links -- in shared memory with TMA bulk copies,
 * two tiles in flight, and compute from there.  It runs where the two-cell kernels run and nx is
 * a multiple of 16 no larger than 512.  Results are bit-identical to the other AA kernels (the
 * force up to the grouping of its partial sums).  Every wait of the kernel on its copies is
 * bounded (2 s); a wait that runs out sets a sticky fault that the next synchronising call
 * (getters, lbm_check_finite) reports as LBM_ETIMEOUT.  Returns 1 when the staged kernel will run,
 * 0 when not, LBM_EINVAL for a NULL context.  Drops the cached step graphs.  ([Layout]'s in-place
 * step; the staging is a GB300 launch choice, not a page's design.) */
int lbm_set_tma_gather(lbm_ctx* ctx, int enable);

/* Run each step's boundary kernel (the special cells: neighbours of MOVING_WALL cells and, in the
 * AA scheme, cells with links across OPEN faces; the A-B pulls take those links, clamped, in their
 * main kernels) beside the step's main kernel (enable != 0, the default) or after it
 * (enable = 0).  Beside: the boundary kernel goes to a private stream of the highest priority,
 * forked from the context stream after the open-face pre-gather and joined back before the next
 * kernel, so lbm_step's ordering on the context stream is unchanged.  It applies to the AA odd
 * step, the A-B pull of the stream layout's one-cell kernels and the AB2 streaming pass, whose
 * main kernels store into no slot of a special cell, so the populations are bit-identical either
 * way; the two-cell A-B pull and the A-B pull of the bundle and collision layouts write those
 * slots (whole-sector stores that the boundary kernel then overwrites) and always run first.  Kernels run one after the other while per-kernel profiling is on.  Returns LBM_OK, LBM_EINVAL for a NULL context; drops
 * the cached step graphs.  (A launch choice for the same update; the per-link rules are
 * [Layout]'s.) */
int lbm_set_boundary_overlap(lbm_ctx* ctx, int enable);

/* Density and velocity of the natural state: rho[N], u[3*N] (fp32).  FLUID: rho = sum f,
 * u = j/rho + g/2 (Guo's half-force shift).  SOLID: 0, 0.  INLET: rho_in, u_in.  MOVING_WALL:
 * 1, u_w.  Synchronous.  ([PortLBM] §3.1: density and momentum are the zeroth and first moments
 * of the populations, v = sum f c; §4: the handler gives access to these macroscopic
 * observables.  The half-force shift is reading R4, as for lbm_set_body_force.) */
int lbm_macroscopic(lbm_ctx* ctx, float* rho, float* u);

/* Force on all SOLID and MOVING_WALL cells (one body) from the last step of the last lbm_step
 * call ([Layout]: the momentum exchange is taken in the step whose forces are read back): the sum
 * over every bounce-back link of a FLUID cell of 2 c_q f*_q (on a MOVING_WALL link
 * c_q (2 f*_q - 6 w_q (c_q.u_w)), what the fluid gives up there), accumulated in fp32 within each
 * warp of 32 cells and in fp64 across warps, in a fixed order.  F[3] in lattice units.
 * LBM_ESTATE before the first step or after the state was reloaded.  Synchronous. */
int lbm_force_momentum_exchange(lbm_ctx* ctx, double F[3]);

/* LBM_OK if every population of every FLUID cell is finite, LBM_ENOTFINITE otherwise.
 * Synchronous. */
int lbm_check_finite(lbm_ctx* ctx);

/* Time steps taken since the last state load (lbm_set_populations / lbm_set_equilibrium). */
int64_t lbm_step_count(lbm_ctx* ctx);

/* Number of this library's kernels launched for this context so far (for accounting). */
int64_t lbm_kernel_launches(lbm_ctx* ctx);

/* Per-kernel timing ([Layout] "Measuring": per-kernel GPU time on request).  enable != 0 records
 * a CUDA event pair around every step kernel launched afterwards; lbm_profile_read returns, for
 * kernel kind `kind` (0 AA even, 1 AA odd, 2 A-B pull, 3 A-B collide, 4 stream, 5 open-face
 * gather, 6 force reduce, 7 boundary kernels of cells next to an inlet or an open face), the
 * number of launches and their summed milliseconds since profiling was enabled, and
 * synchronises the stream.  The environment variable LBM_PROFILE=1 at lbm_create turns
 * profiling on from the start.  While it is on, steps are launched one by one (no graphs). */
int lbm_profile_enable(lbm_ctx* ctx, int enable);
int lbm_profile_read(lbm_ctx* ctx, int kind, int64_t* launches, double* total_ms);

/* Release every resource of the context.  NULL-safe.  Synchronises its stream first; the
 * caller's stream itself is not destroyed.  (No page: the counterpart of lbm_create in this
 * ABI's own lifetime convention.) */
void lbm_destroy(lbm_ctx* ctx);

/* ---- slab decomposition along z (several contexts, one per rank) ----------------------------------
 * [Disaggregated] ("Disaggregated Design for GPU-Based Volumetric Data Structures", section
 * "Improving LBM Scalability"): the domain is split into slabs along one axis, and each slab
 * exchanges its boundary data with its two neighbours every time step.  A rank's context holds its
 * owned planes plus one GHOST plane below (z = 0) and one above (z = nz - 1), copies of the
 * neighbouring slabs' boundary planes.  After every lbm_step(ctx, 1) the rank packs what its
 * neighbours need (lbm_halo_pack), the ranks swap those buffers, and each unpacks what it received
 * into its ghost planes (lbm_halo_unpack).  Only the five populations that cross a slab face are
 * exchanged: 10 nx ny values per slab and step.  The force of lbm_force_momentum_exchange then
 * covers the owned cells only; the ranks add theirs.  The host side (partition, neighbours,
 * message order, force reduction) is lattice_boltzmann_cfd_d3q19_gb300/slab.py. */

/* enable != 0: planes z = 0 and z = nz - 1 of this context become ghost planes.  Their cells are
 * stepped like the others, but their results are replaced by lbm_halo_unpack.  They have no links
 * for the momentum exchange and are never special.  Needs the A-B scheme (LBM_STREAMING_AB),
 * PERIODIC z faces and nz >= 3; LBM_EINVAL otherwise.  While enabled, lbm_step accepts n <= 1 only,
 * and lbm_set_faces keeps z PERIODIC.  Flags, populations and fields of the ghost planes are set
 * and read like any others: load them with the neighbours' boundary planes.  Synchronous; drops
 * the cached step graphs. */
int lbm_set_ghost_planes(lbm_ctx* ctx, int enable);

/* Elements of one halo buffer: 5 nx ny (-1 for a NULL context). */
int64_t lbm_halo_elements(lbm_ctx* ctx);
/* Bytes of one halo element: the internal storage of the populations (4; 2 in half-precision
 * storage).  Halo buffers are opaque: they hold stored values, meaningful only to lbm_halo_unpack
 * of a context with the same layout. */
int lbm_halo_element_bytes(lbm_ctx* ctx);

/* After a step: the post-collision populations with c_z = -1 of the first owned plane (z = 1) into
 * lo, and those with c_z = +1 of the last owned plane (z = nz - 2) into hi.  Each buffer holds
 * lbm_halo_elements values, population-major in q order, cell x + nx y within a population.  lo
 * goes to the slab below, hi to the slab above.  lo and hi are device memory of the current
 * device (LBM_EINVAL otherwise).  LBM_ESTATE without ghost planes, or before the first step after
 * a state load.  Asynchronous on the context stream. */
int lbm_halo_pack(lbm_ctx* ctx, void* lo, void* hi);

/* Write the neighbours' buffers into the ghost planes: from_below (the hi of the slab below) into
 * the c_z = +1 populations of plane z = 0, and from_above (the lo of the slab above) into the
 * c_z = -1 populations of plane z = nz - 1.  These are the only ghost values the next step's pull
 * reads.  Same requirements and errors as lbm_halo_pack; asynchronous. */
int lbm_halo_unpack(lbm_ctx* ctx, const void* from_below, const void* from_above);

/* One step of a slab with its halo exchange overlapped by the interior planes.  [Disaggregated],
 * section "Disaggregation on a Dense Domain" (Overlapping Computation and Communication, OCC) and
 * "Improving LBM Scalability", "Reference Implementation": a stencil step is split into the voxels
 * that only need local data and the voxels that need the neighbours' data, so that the halo
 * travels while the first kind is computed.  For a pull step the order is: the two boundary
 * planes, whose results the neighbours need, then the interior while their halo travels.  A
 * step = lbm_slab_step_begin, the exchange of lo / hi by the caller, then lbm_slab_step_end.
 * Results are bit for bit those of lbm_step(ctx, 1) + lbm_halo_pack + exchange + lbm_halo_unpack.
 * The force is summed in another order, so it agrees to rounding only.
 *
 * lbm_slab_step_begin: on the context stream, steps the owned boundary planes z = 1 and
 * z = nz - 2 and their special cells, then packs their outgoing populations into lo and hi (as
 * lbm_halo_pack).  It then launches the interior planes 2 .. nz - 3 and their special cells on the
 * context's side stream, which waits for the pack.  A transfer the caller enqueues after this call,
 * ordered after the context stream, therefore runs beside the interior.  The ghost planes are not
 * stepped.  lo and hi are device memory of the current device (LBM_EINVAL otherwise).  LBM_ESTATE
 * without ghost planes, or with a slab step already open.  Asynchronous. */
int lbm_slab_step_begin(lbm_ctx* ctx, void* lo, void* hi);

/* lbm_slab_step_end: the context stream waits for the interior planes, the step is completed (the
 * momentum exchange of the owned cells, the buffer swap, the step count), and from_below /
 * from_above are unpacked into the ghost planes (as lbm_halo_unpack).  The caller orders the
 * receipt of the buffers before this call on the context stream (a communication library's wait
 * on the stream).  LBM_ESTATE when no slab step is open.  Between begin and end, every other call
 * on the context except lbm_halo_elements, lbm_halo_element_bytes, lbm_step_count,
 * lbm_kernel_launches and lbm_destroy returns LBM_ESTATE.  Asynchronous. */
int lbm_slab_step_end(lbm_ctx* ctx, const void* from_below, const void* from_above);

/* Momentum-exchange force of ONE collision of a caller-held state, without allocating any memory.
 * The source papers and pages describe no counterpart to this entry point.  It exists for callers
 * that cannot call cudaMalloc: plug-ins whose host application owns all device memory through its
 * own pool (an allocation behind the pool's back can fail or break its accounting), and tools that
 * must not grow the footprint of a process they are embedded in.  It computes what
 * lbm_force_momentum_exchange reports after lbm_set_populations(f) and lbm_step(1) on a context
 * with the same grid, tau, flags, faces and body force: the sum over every bounce-back link of a
 * FLUID cell of 2 c_q f*_q, f* the post-collision state.
 *   f       device memory, canonical natural state f[q*N + n] (absolute fp32), 19*N floats;
 *   flags   device memory, N bytes, LBM_FLUID / LBM_SOLID / LBM_INLET (LBM_MOVING_WALL and other
 *           values -> LBM_EINVAL, F unchanged);
 *   face_*  LBM_PERIODIC or LBM_OPEN per axis; tau > 1/2; g the body acceleration (Guo forcing);
 *   F       host memory, 3 doubles, written on success;
 *   cuda_stream  the stream to run on (NULL: the legacy default stream); synchronised on return.
 * f, flags and the stream must belong to the CUDA device that is current on the calling thread;
 * f or flags on another device -> LBM_EINVAL.
 * Working memory: one fixed array of about 1.5 MiB in the library's static device memory, held
 * by every GPU that loads the library until the process exits.  Grids of more than 16,777,216
 * cells (256^3) exceed it and are rejected with LBM_EINVAL before any CUDA call.  The first call
 * on each device looks the array's device address up (cudaGetSymbolAddress); make that first
 * call before any stream capture.  All calls share the array and each clears what it reads
 * before writing it: calls that overlap on the GPU (on different streams or host threads) race
 * and give wrong results; serialise them. */
int lbm_force_momentum_exchange_noalloc(const float* f, const uint8_t* flags, int nx, int ny,
                                        int nz, int face_x, int face_y, int face_z, float tau,
                                        float gx, float gy, float gz, double F[3],
                                        void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* LBM_H */
