// D3Q19 BGK lattice Boltzmann -- CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
//
// This file is the plain, slow, double-precision statement of what the GPU library computes.  It
// is used by the tests, by the smoke check and by the benchmark's CPU-baseline leg, and by nothing
// else.  It shares no code, header, table or helper with the CUDA library: its velocity set,
// weights, opposite table, equilibrium, forcing and boundary rules are all written out here again.
//
// Sources (page title, then section / equation):
//  * "PortLBM: A Portable Lattice Boltzmann Tool Leveraging SYCL on AMD, NVIDIA, and Intel GPUs",
//    §3.1 Eq. 1 (BGK lattice Boltzmann equation, time step 1), §3.3 Eq. 3 (split into a collision
//    and a streaming step; one-step pull two-lattice scheme), §3.1 last paragraph (equilibrium
//    inlet, halfway bounce-back, Neumann-type outlet).
//  * "GPU lattice Boltzmann: streaming layout and performance", the "In place" and "Two buffers"
//    bullets (AA addressing; two-buffer collide-then-pull) and the paragraph after them (the same
//    per-link rules in both layouts; momentum exchange on the last step of a submission).
//  * "GPU加速LBM流体仿真：从原理到150倍性能优化实战", §2.2 (D3Q19 weights 1/3, 1/18, 1/36) and
//    §5.1 (omega = 1/(3 nu + 1/2)).
//
// Readings taken where the pages are silent (each is listed in the design notes):
//  * equilibrium: the compressible second-order form w rho [1 + 3 c.u + 9/2 (c.u)^2 - 3/2 u.u]
//    with u = j / rho (PortLBM prints the incompressible 2D variant of the same polynomial);
//  * body force: Guo forcing with F = rho g, the half-force velocity shift u = j/rho + g/2 and
//    the source term (1 - omega/2) w [3 (c - u).F + 9 (c.u)(c.F)];
//  * SOLID cells reflect (halfway bounce-back), INLET cells are fixed reservoirs at
//    f_eq(rho_in, u_in), an OPEN face is zero-gradient: a population whose source lies beyond the
//    face is taken from the source clamped onto the last layer of that axis;
//  * MOVING_WALL cells reflect like SOLID ones plus the moving-wall term of the mirror method
//    ("GPU加速LBM流体仿真", §4.2): 2 w_q rho (c_q.u_w) / c_s^2 with rho the reference density 1;
//  * momentum exchange on the solid: sum over bounce-back links of 2 c_q f*_q (f* = post-collision),
//    and on a moving-wall link c_q (2 f*_q - 6 w_q (c_q.u_w)) (what the fluid gives up there).
//
// Parity pins: every function here is checked by tests/test_oracle_pins.py against closed forms,
// invariants and brute force (weights and moments, equilibrium fixed point, exact conservation,
// Taylor-Green decay, Poiseuille profile, AA == two-lattice, streaming permutation).
//
// Build: g++ -O2 -std=c++17 -fopenmp -ffp-contract=off -shared -fPIC (no fused multiply-add, so
// results do not depend on the host's instruction set).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---- velocity set (GPU加速LBM §2.2: rest, 6 axis, 12 edge diagonals) --------------------------
// Member order: each moving velocity is followed by its opposite.
const int C[19][3] = {
    {0, 0, 0},
    {1, 0, 0},  {-1, 0, 0}, {0, 1, 0},  {0, -1, 0}, {0, 0, 1},   {0, 0, -1},
    {1, 1, 0},  {-1, -1, 0}, {1, 0, 1}, {-1, 0, -1}, {0, 1, 1},  {0, -1, -1},
    {1, -1, 0}, {-1, 1, 0}, {1, 0, -1}, {-1, 0, 1}, {0, 1, -1}, {0, -1, 1}};

double weight(int q) {
    int speed2 = C[q][0] * C[q][0] + C[q][1] * C[q][1] + C[q][2] * C[q][2];
    if (speed2 == 0) return 1.0 / 3.0;
    if (speed2 == 1) return 1.0 / 18.0;
    return 1.0 / 36.0;
}

// opposite(q): the member whose velocity is -c_q, found by search (no hand-written table).
int opposite(int q) {
    for (int p = 0; p < 19; ++p)
        if (C[p][0] == -C[q][0] && C[p][1] == -C[q][1] && C[p][2] == -C[q][2]) return p;
    return -1;
}

enum { FLUID = 0, SOLID = 1, INLET = 2, MOVING_WALL = 3 };
enum { PERIODIC = 0, OPEN = 1 };

struct Grid {
    int n[3];
    int face[3];
    int64_t N;
    int64_t cell(const int x[3]) const {
        return (int64_t)x[0] + (int64_t)n[0] * ((int64_t)x[1] + (int64_t)n[1] * (int64_t)x[2]);
    }
};

// Neighbour of x displaced by d (d in {-1,0,1}^3).  Periodic axes wrap.  On an OPEN axis a
// coordinate beyond the face is clamped onto the last layer (the zero-gradient ghost equals it);
// *beyond reports whether any axis was clamped.
void displaced(const Grid& g, const int x[3], const int d[3], int s[3], bool* beyond) {
    *beyond = false;
    for (int a = 0; a < 3; ++a) {
        int v = x[a] + d[a];
        if (v < 0 || v >= g.n[a]) {
            if (g.face[a] == PERIODIC) {
                v = ((v % g.n[a]) + g.n[a]) % g.n[a];
            } else {
                v = v < 0 ? 0 : g.n[a] - 1;
                *beyond = true;
            }
        }
        s[a] = v;
    }
}

// Second-order equilibrium, c_s^2 = 1/3.
void equilibrium(double rho, const double u[3], double feq[19]) {
    double uu = u[0] * u[0] + u[1] * u[1] + u[2] * u[2];
    for (int q = 0; q < 19; ++q) {
        double cu = C[q][0] * u[0] + C[q][1] * u[1] + C[q][2] * u[2];
        feq[q] = weight(q) * rho * (1.0 + 3.0 * cu + 4.5 * cu * cu - 1.5 * uu);
    }
}

// BGK collision with Guo forcing (PortLBM §3.1 Eq. 1 right-hand side; forcing: reading above).
void collide(const double f[19], double omega, const double g[3], double post[19]) {
    double rho = 0.0, j[3] = {0.0, 0.0, 0.0};
    for (int q = 0; q < 19; ++q) {
        rho += f[q];
        for (int a = 0; a < 3; ++a) j[a] += f[q] * C[q][a];
    }
    double u[3], F[3];
    for (int a = 0; a < 3; ++a) {
        u[a] = j[a] / rho + 0.5 * g[a];
        F[a] = rho * g[a];
    }
    double feq[19];
    equilibrium(rho, u, feq);
    double uF = u[0] * F[0] + u[1] * F[1] + u[2] * F[2];
    for (int q = 0; q < 19; ++q) {
        double cu = C[q][0] * u[0] + C[q][1] * u[1] + C[q][2] * u[2];
        double cF = C[q][0] * F[0] + C[q][1] * F[1] + C[q][2] * F[2];
        double Fq = (1.0 - 0.5 * omega) * weight(q) * (3.0 * (cF - uF) + 9.0 * cu * cF);
        post[q] = f[q] - omega * (f[q] - feq[q]) + Fq;
    }
}

struct Problem {
    Grid grid;
    double omega;
    double g[3];
    double feq_in[19];
    double uw[3];  // velocity of the MOVING_WALL cells
    const uint8_t* flags;
};

// Moving-wall term of a link whose population q leaves the wall toward the fluid: the mirror
// method's 2 w_q rho (c_q.u_w) / c_s^2 with c_s^2 = 1/3 and the reference density 1.
double wall_term(const Problem& P, int q) {
    double cu = C[q][0] * P.uw[0] + C[q][1] * P.uw[1] + C[q][2] * P.uw[2];
    return 6.0 * weight(q) * cu;
}

int setup(Problem* P, int nx, int ny, int nz, double tau, const uint8_t* flags, const int* faces,
          const double* inlet, const double* g, const double* wall) {
    if (nx < 1 || ny < 1 || nz < 1 || !(tau > 0.5) || !flags || !faces) return -1;
    P->grid.n[0] = nx;
    P->grid.n[1] = ny;
    P->grid.n[2] = nz;
    P->grid.N = (int64_t)nx * ny * nz;
    for (int a = 0; a < 3; ++a) {
        if (faces[a] != PERIODIC && faces[a] != OPEN) return -1;
        P->grid.face[a] = faces[a];
    }
    for (int64_t n = 0; n < P->grid.N; ++n)
        if (flags[n] > MOVING_WALL) return -1;
    P->omega = 1.0 / tau;
    for (int a = 0; a < 3; ++a) P->g[a] = g ? g[a] : 0.0;
    double rho_in = inlet ? inlet[0] : 1.0;
    double u_in[3] = {inlet ? inlet[1] : 0.0, inlet ? inlet[2] : 0.0, inlet ? inlet[3] : 0.0};
    equilibrium(rho_in, u_in, P->feq_in);
    for (int a = 0; a < 3; ++a) P->uw[a] = wall ? wall[a] : 0.0;
    P->flags = flags;
    return 0;
}

void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

// Momentum given to SOLID cells by the post-collision state `post` (natural SoA, indexed
// post[q*N + n]): every link of a FLUID cell x along which population q bounces back carries
// 2 c_q f*_q(x).  Population q of x bounces back when the cell it would stream into (x + c_q,
// wrapped or clamped like any source) is SOLID.  Summed per z-plane, then over planes in order, so
// the result does not depend on the thread count.
void momentum_exchange(const Problem& P, const double* post, double force[3]) {
    const Grid& G = P.grid;
    std::vector<double> plane(3 * (size_t)G.n[2], 0.0);
#pragma omp parallel for schedule(static)
    for (int z = 0; z < G.n[2]; ++z) {
        double acc[3] = {0.0, 0.0, 0.0};
        for (int y = 0; y < G.n[1]; ++y)
            for (int x = 0; x < G.n[0]; ++x) {
                int X[3] = {x, y, z};
                int64_t n = G.cell(X);
                if (P.flags[n] != FLUID) continue;
                for (int q = 1; q < 19; ++q) {
                    int s[3];
                    bool beyond;
                    displaced(G, X, C[q], s, &beyond);
                    uint8_t partner = P.flags[G.cell(s)];
                    if (partner != SOLID && partner != MOVING_WALL) continue;
                    double fq = post[(int64_t)q * G.N + n];
                    // what the fluid gives up: f*_q leaves, the reflected population returns
                    double back = partner == SOLID ? fq : fq + wall_term(P, opposite(q));
                    for (int a = 0; a < 3; ++a) acc[a] += C[q][a] * (fq + back);
                }
            }
        for (int a = 0; a < 3; ++a) plane[3 * (size_t)z + a] = acc[a];
    }
    for (int a = 0; a < 3; ++a) force[a] = 0.0;
    for (int z = 0; z < G.n[2]; ++z)
        for (int a = 0; a < 3; ++a) force[a] += plane[3 * (size_t)z + a];
}

// Incoming population q at FLUID cell X, taken from a post-collision state through the per-link
// rules.  `post_at(q, n)` returns post-collision population q of cell n.
template <class PostAt>
double incoming(const Problem& P, const int X[3], int q, PostAt post_at) {
    const Grid& G = P.grid;
    int d[3] = {-C[q][0], -C[q][1], -C[q][2]};
    int s[3];
    bool beyond;
    displaced(G, X, d, s, &beyond);
    int64_t ns = G.cell(s);
    switch (P.flags[ns]) {
        case FLUID: return post_at(q, ns);                     // streamed from the source
        case SOLID: return post_at(opposite(q), G.cell(X));   // halfway bounce-back
        case MOVING_WALL:                                      // bounce-back off a moving wall
            return post_at(opposite(q), G.cell(X)) + wall_term(P, q);
        default: return P.feq_in[q];                          // equilibrium reservoir
    }
}

}  // namespace

extern "C" {

// Velocity set, weights and opposite table, for the tests.
void oracle_tables(int* c, double* w, int* opp) {
    for (int q = 0; q < 19; ++q) {
        for (int a = 0; a < 3; ++a) c[3 * q + a] = C[q][a];
        w[q] = weight(q);
        opp[q] = opposite(q);
    }
}

void oracle_equilibrium(double rho, const double* u, double* feq) { equilibrium(rho, u, feq); }

// One cell's collision: f (19) -> post (19), relaxation omega = 1/tau, body acceleration g.
void oracle_collide(const double* f, double tau, const double* g, double* post) {
    double zero[3] = {0.0, 0.0, 0.0};
    collide(f, 1.0 / tau, g ? g : zero, post);
}

// Equilibrium populations for whole fields: rho[N], u[3][N] -> f[19][N] (natural SoA).
void oracle_equilibrium_field(int64_t N, const double* rho, const double* u, double* f) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double uu[3] = {u[n], u[N + n], u[2 * N + n]}, feq[19];
        equilibrium(rho[n], uu, feq);
        for (int q = 0; q < 19; ++q) f[(int64_t)q * N + n] = feq[q];
    }
}

// Two-lattice step, the definition (PortLBM §3.3: collision, then one-step pull into a second
// lattice; per-link rules as listed at the top of this file).
//   f      : natural populations f[q*N + n], n = x + nx*(y + ny*z); updated in place.
//   flags  : N bytes, 0 FLUID / 1 SOLID / 2 INLET.  Only FLUID cells are updated.
//   faces  : 3 ints, 0 PERIODIC / 1 OPEN, per axis.
//   inlet  : rho_in, ux, uy, uz (may be NULL: rho 1, u 0).   g: body acceleration (may be NULL).
//   force  : if not NULL, momentum exchange of the last step's post-collision state.
// Returns 0, or -1 on invalid arguments.
int oracle_step_ab(int nx, int ny, int nz, double tau, const uint8_t* flags, const int* faces,
                   const double* inlet, const double* g, const double* wall, double* f,
                   int nsteps, double* force, int nthreads) {
    Problem P;
    if (setup(&P, nx, ny, nz, tau, flags, faces, inlet, g, wall) != 0 || nsteps < 0 || !f)
        return -1;
    set_threads(nthreads);
    const Grid& G = P.grid;
    const int64_t N = G.N;
    std::vector<double> post((size_t)(19 * N), 0.0);
    if (force) force[0] = force[1] = force[2] = 0.0;
    for (int step = 0; step < nsteps; ++step) {
        // collision
#pragma omp parallel for schedule(static)
        for (int z = 0; z < G.n[2]; ++z)
            for (int y = 0; y < G.n[1]; ++y)
                for (int x = 0; x < G.n[0]; ++x) {
                    int X[3] = {x, y, z};
                    int64_t n = G.cell(X);
                    if (flags[n] != FLUID) continue;
                    double fn[19], pn[19];
                    for (int q = 0; q < 19; ++q) fn[q] = f[(int64_t)q * N + n];
                    collide(fn, P.omega, P.g, pn);
                    for (int q = 0; q < 19; ++q) post[(size_t)((int64_t)q * N + n)] = pn[q];
                }
        if (force && step == nsteps - 1) momentum_exchange(P, post.data(), force);
        // streaming (pull) into f: every FLUID cell's populations come from `post` only
        auto post_at = [&](int q, int64_t n) { return post[(size_t)((int64_t)q * N + n)]; };
#pragma omp parallel for schedule(static)
        for (int z = 0; z < G.n[2]; ++z)
            for (int y = 0; y < G.n[1]; ++y)
                for (int x = 0; x < G.n[0]; ++x) {
                    int X[3] = {x, y, z};
                    int64_t n = G.cell(X);
                    if (flags[n] != FLUID) continue;
                    for (int q = 0; q < 19; ++q) f[(int64_t)q * N + n] = incoming(P, X, q, post_at);
                }
    }
    return 0;
}

// In-place AA step on ONE buffer A[q*N + n] ("GPU lattice Boltzmann: streaming layout and
// performance", "In place" bullet).  `parity` is the number of steps already taken mod 2.
//  even step: read population q of x at (q, x); write the collided one at (opposite(q), x).
//  odd step : read it at (opposite(q), x - c_q); write it at (q, x + c_q).
// Boundary links follow the same per-link rules as the two-lattice step, applied at the cell's
// own slots: a link whose partner cell is SOLID or INLET reads or writes the cell's own mirrored
// slot, and open-face (zero-gradient) copies are filled from the post-collision state after the
// scatter.  As that page describes, the odd step gathers every link into scratch before any write.
// After an odd number of total steps the buffer holds post-collision values at (opposite(q), x);
// oracle_aa_natural() turns that into natural populations.
int oracle_step_aa(int nx, int ny, int nz, double tau, const uint8_t* flags, const int* faces,
                   const double* inlet, const double* g, const double* wall, double* A,
                   int parity, int nsteps, double* force, int nthreads) {
    Problem P;
    if (setup(&P, nx, ny, nz, tau, flags, faces, inlet, g, wall) != 0 || nsteps < 0 || !A ||
        (parity != 0 && parity != 1))
        return -1;
    set_threads(nthreads);
    const Grid& G = P.grid;
    const int64_t N = G.N;
    auto slot = [&](int q, int64_t n) -> double& { return A[(int64_t)q * N + n]; };
    std::vector<double> post((size_t)(19 * N), 0.0);
    if (force) force[0] = force[1] = force[2] = 0.0;
    for (int step = 0; step < nsteps; ++step, parity ^= 1) {
        bool last = force && step == nsteps - 1;
        if (parity == 0) {
            for (int z = 0; z < G.n[2]; ++z)
                for (int y = 0; y < G.n[1]; ++y)
                    for (int x = 0; x < G.n[0]; ++x) {
                        int X[3] = {x, y, z};
                        int64_t n = G.cell(X);
                        if (flags[n] != FLUID) continue;
                        double fn[19], pn[19];
                        for (int q = 0; q < 19; ++q) fn[q] = slot(q, n);
                        collide(fn, P.omega, P.g, pn);
                        for (int q = 0; q < 19; ++q) {
                            slot(opposite(q), n) = pn[q];
                            post[(size_t)((int64_t)q * N + n)] = pn[q];
                        }
                    }
            if (last) momentum_exchange(P, post.data(), force);
            continue;
        }
        // odd step, gather pass: incoming populations of every FLUID cell, from the even step's
        // post-collision values, which sit at (opposite(q), x).
        std::vector<double> gathered((size_t)(19 * N), 0.0);
        auto even_post_at = [&](int q, int64_t n) { return slot(opposite(q), n); };
        for (int z = 0; z < G.n[2]; ++z)
            for (int y = 0; y < G.n[1]; ++y)
                for (int x = 0; x < G.n[0]; ++x) {
                    int X[3] = {x, y, z};
                    int64_t n = G.cell(X);
                    if (flags[n] != FLUID) continue;
                    for (int q = 0; q < 19; ++q)
                        gathered[(size_t)((int64_t)q * N + n)] = incoming(P, X, q, even_post_at);
                }
        // collision
        for (int64_t n = 0; n < N; ++n) {
            if (flags[n] != FLUID) continue;
            double fn[19], pn[19];
            for (int q = 0; q < 19; ++q) fn[q] = gathered[(size_t)((int64_t)q * N + n)];
            collide(fn, P.omega, P.g, pn);
            for (int q = 0; q < 19; ++q) post[(size_t)((int64_t)q * N + n)] = pn[q];
        }
        if (last) momentum_exchange(P, post.data(), force);
        // scatter pass: post-collision population q of x goes to (q, x + c_q)
        for (int z = 0; z < G.n[2]; ++z)
            for (int y = 0; y < G.n[1]; ++y)
                for (int x = 0; x < G.n[0]; ++x) {
                    int X[3] = {x, y, z};
                    int64_t n = G.cell(X);
                    if (flags[n] != FLUID) continue;
                    for (int q = 0; q < 19; ++q) {
                        double pq = post[(size_t)((int64_t)q * N + n)];
                        int p = opposite(q);
                        int d[3];
                        bool beyond;
                        displaced(G, X, C[q], d, &beyond);
                        uint8_t fd = flags[G.cell(d)];
                        if (!beyond && fd == FLUID) {
                            slot(q, G.cell(d)) = pq;              // streamed to the neighbour
                        } else if (fd == SOLID) {
                            slot(p, n) = pq;                       // bounced back into x
                        } else if (fd == MOVING_WALL) {
                            slot(p, n) = pq + wall_term(P, p);     // off the moving wall
                        } else if (fd == INLET) {
                            slot(p, n) = P.feq_in[p];              // reservoir feeds x
                        }
                        // beyond an open face with a FLUID clamped partner: filled below
                    }
                }
        // open-face fill: population q of a FLUID cell r whose source lies beyond an open face
        // is the clamped source's post-collision population q (zero-gradient ghost).
        for (int z = 0; z < G.n[2]; ++z)
            for (int y = 0; y < G.n[1]; ++y)
                for (int x = 0; x < G.n[0]; ++x) {
                    int X[3] = {x, y, z};
                    int64_t n = G.cell(X);
                    if (flags[n] != FLUID) continue;
                    for (int q = 0; q < 19; ++q) {
                        int d[3] = {-C[q][0], -C[q][1], -C[q][2]}, s[3];
                        bool beyond;
                        displaced(G, X, d, s, &beyond);
                        int64_t ns = G.cell(s);
                        if (beyond && flags[ns] == FLUID)
                            slot(q, n) = post[(size_t)((int64_t)q * N + ns)];
                    }
                }
    }
    return 0;
}

// Natural populations from an AA buffer after an odd number of steps (post-collision values at
// (opposite(q), x)): the streaming half of the next odd step, without its collision.
// Non-FLUID cells are copied unchanged.
int oracle_aa_natural(int nx, int ny, int nz, const uint8_t* flags, const int* faces,
                      const double* inlet, const double* wall, const double* A, double* f) {
    Problem P;
    if (setup(&P, nx, ny, nz, 1.0, flags, faces, inlet, nullptr, wall) != 0 || !A || !f)
        return -1;
    const Grid& G = P.grid;
    const int64_t N = G.N;
    auto post_at = [&](int q, int64_t n) { return A[(int64_t)opposite(q) * N + n]; };
    for (int z = 0; z < G.n[2]; ++z)
        for (int y = 0; y < G.n[1]; ++y)
            for (int x = 0; x < G.n[0]; ++x) {
                int X[3] = {x, y, z};
                int64_t n = G.cell(X);
                for (int q = 0; q < 19; ++q)
                    f[(int64_t)q * N + n] =
                        flags[n] == FLUID ? incoming(P, X, q, post_at) : A[(int64_t)q * N + n];
            }
    return 0;
}

// Density and velocity of a natural state.  FLUID: rho = sum f, u = j/rho + g/2 (Guo's
// half-force shift).  SOLID: 0, 0.  INLET: rho_in, u_in.  MOVING_WALL: 1, u_w.
// rho[N], u[3][N].
int oracle_macroscopic(int nx, int ny, int nz, const uint8_t* flags, const double* inlet,
                       const double* wall, const double* g, const double* f, double* rho,
                       double* u) {
    if (nx < 1 || ny < 1 || nz < 1 || !flags || !f || !rho || !u) return -1;
    const int64_t N = (int64_t)nx * ny * nz;
    double gg[3] = {g ? g[0] : 0.0, g ? g[1] : 0.0, g ? g[2] : 0.0};
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        if (flags[n] == SOLID) {
            rho[n] = 0.0;
            u[n] = u[N + n] = u[2 * N + n] = 0.0;
        } else if (flags[n] == INLET) {
            rho[n] = inlet ? inlet[0] : 1.0;
            for (int a = 0; a < 3; ++a) u[a * N + n] = inlet ? inlet[1 + a] : 0.0;
        } else if (flags[n] == MOVING_WALL) {
            rho[n] = 1.0;
            for (int a = 0; a < 3; ++a) u[a * N + n] = wall ? wall[a] : 0.0;
        } else {
            double r = 0.0, j[3] = {0.0, 0.0, 0.0};
            for (int q = 0; q < 19; ++q) {
                double fq = f[(int64_t)q * N + n];
                r += fq;
                for (int a = 0; a < 3; ++a) j[a] += fq * C[q][a];
            }
            rho[n] = r;
            for (int a = 0; a < 3; ++a) u[a * N + n] = j[a] / r + 0.5 * gg[a];
        }
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

}  // extern "C"
