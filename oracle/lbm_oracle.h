/*
 * lbm_oracle.h -- plain fp64 CPU oracle for the lattice-Boltzmann collide-and-stream step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or call this
 * library; only tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (one time step, for every fluid cell, in this order):
 *   moments -> force -> equilibria -> Guo source -> collision (BGK or MRT, and the
 *   thermal MRT) -> pull streaming into a second buffer with half-way bounce-back /
 *   anti-bounce-back on wall links -> momentum exchange on solid links.
 * Sources: "Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI"
 * (Sec. 2, Eq. 5 and Eq. 7 with the bounce-back and anti-bounce-back rules below them);
 * "GPU Optimization for High-Quality Kinetic Fluid Simulation" (Sec. 3.1, Eq. 1-5);
 * "GPU lattice Boltzmann: streaming layout and performance" (two-buffer scheme: collide,
 * then pull into the other buffer).
 *
 * D3Q27 central-moment MRT ("GPU Optimization for High-Quality Kinetic Fluid Simulation",
 * Sec. 3.1 Eq. 5 with the D3Q27 lattice of Fig. 2, fixed rates): the moments are the 27
 * central moments prod_a (c_a - u_a)^e_a, e in {0,1,2}^3, with the three second-order
 * normal moments recombined as xx - yy, xx - zz (shear) and xx + yy + zz (bulk); the
 * equilibrium is the product form f_eq = rho prod_a phi(c_a, u_a) whose central moments are
 * rho prod_a (1, 0, 1/3)[e_a]; the force source is (F/rho) . d f_eq / du.
 *
 * Layout: structure of arrays, x fastest: f[q*W + i + wx*(j + wy*k)] where W = wx*wy*wz is
 * the number of cells the run holds (a window of the whole nx*ny*nz domain; the window is
 * the whole domain in an ordinary run).  A population whose pull source lies inside the
 * domain but outside the window is unknown and is set to NaN, so that a window run yields
 * exact values only at cells further from the window's cut faces than the number of steps.
 */
#ifndef LBM_ORACLE_H
#define LBM_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_D2Q9 = 9, ORC_D3Q19 = 19, ORC_D3Q27 = 27 };
enum { ORC_THERMAL_NONE = 0, ORC_D2Q5 = 5, ORC_D3Q7 = 7 };
enum { ORC_BGK = 0, ORC_MRT = 1, ORC_CM = 2 };
enum { ORC_PERIODIC = 0, ORC_WALL = 1 };
enum { ORC_ADIABATIC = 0, ORC_DIRICHLET = 1 };

typedef struct {
    int lattice;          /* ORC_D2Q9, ORC_D3Q19 or ORC_D3Q27 */
    int thermal;          /* ORC_THERMAL_NONE, ORC_D2Q5 (with D2Q9), ORC_D3Q7 (with D3Q19) */
    int collision;        /* ORC_BGK or ORC_MRT (D2Q9, D3Q19); ORC_CM (D3Q27) */
    double tau;           /* BGK relaxation time; CM: 1/tau is the shear rate */
    double s[19];         /* MRT rate of each moment row; rows of conserved moments ignored */
    double s_T[7];        /* thermal MRT rate of each row; row 0 (T) ignored */
    double cm_rates[5];   /* CM rates: trace of the second-order moments (bulk), then the
                             third-, fourth-, fifth- and sixth-order central moments */
    double a_T;           /* thermal energy-moment constant: e_eq = a_T * T */
    double g_body[3];     /* body acceleration: F += rho * g_body */
    double gbeta;         /* buoyancy: F += rho * gbeta * (T - T0) along up_axis */
    double T0;
    int up_axis;          /* 0, 1, 2 = x, y, z */
    int face_flow[6];     /* per face (-x,+x,-y,+y,-z,+z): ORC_PERIODIC or ORC_WALL */
    int face_T[6];        /* on WALL faces: ORC_ADIABATIC or ORC_DIRICHLET */
    double T_wall[6];     /* wall temperature of DIRICHLET faces */
    int nx, ny, nz;       /* whole domain (nz == 1 for D2Q9) */
    int x0, y0, z0;       /* window origin in the domain */
    int wx, wy, wz;       /* window extent */
    const unsigned char *solid;   /* wx*wy*wz flags, 1 = solid cell; NULL = no solid */
    /* immersed boundary ("GPU Optimization for High-Quality Kinetic Fluid Simulation",
     * Sec. 3.1, Eq. 6-8): ib_n samples at ib_x (3 per sample, domain coordinates, cell
     * centres at integers) with boundary velocity ib_ub (3 per sample, NULL = 0) and weight
     * ib_w (NULL = 1).  Each step: trilinear (bilinear in 2-D) interpolation of rho and
     * u = (j + F_body/2)/rho at the samples from the pre-collision state, penalty
     * g = w rho (u_b - u), spread with the same kernel into a per-cell force added to the
     * body force of that step's collision. */
    int ib_n;
    const double *ib_x, *ib_ub, *ib_w;
} oracle_problem;

/* 0 on success, negative on a bad problem description. */
int oracle_check(const oracle_problem *p);

/* f = f_eq(rho, u), g = g_eq(T, u) (moment form) in every fluid cell; solid cells get 0.
 * rho: W, u: 3*W (component-major; the z part is ignored in 2D), T: W or NULL. */
int oracle_init_equilibrium(const oracle_problem *p, const double *rho, const double *u,
                            const double *T, double *f, double *g);

/* One step.  f, g hold the state at t on entry and at t+1 on return.  fpost, gpost are
 * scratch buffers of the same size (post-collision values).  force[3] receives the
 * momentum exchanged with solid-mask cells during this step (may be NULL); ib[6] the
 * immersed boundary's reaction force -sum g and its torque about the samples' centroid
 * (may be NULL). */
int oracle_step(const oracle_problem *p, double *f, double *g, double *fpost, double *gpost,
                double force[3], double ib[6]);

/* steps repeated oracle_step calls; allocates its own scratch. force, ib: last step's. */
int oracle_run(const oracle_problem *p, double *f, double *g, int steps, double force[3],
               double ib[6]);

/* The immersed-boundary force per cell (3 planes of W) the next step would add, and
 * ib[6] as in oracle_step (for tests of the interpolation and spreading). */
int oracle_ib_forces(const oracle_problem *p, const double *f, const double *g, double *Fib,
                     double ib[6]);

/* rho = sum f, u = (sum c f + F/2) / rho, T = sum g; solid cells read as 0. */
int oracle_macroscopic(const oracle_problem *p, const double *f, const double *g, double *rho,
                       double *u, double *T);

/* out[0] mass = sum rho, out[1..3] momentum = sum c f over fluid cells,
 * out[4..9] per face: sum over fluid cells next to a DIRICHLET face of 2 (T_w - T_cell),
 * out[10..12]: sum over fluid cells of u_a T with u = (j + F/2)/rho (0 without thermal). */
int oracle_diagnostics(const oracle_problem *p, const double *f, const double *g,
                       double out[13]);

/* The lattice tables the oracle uses, for inspection by tests.  kind = 9, 19 (momentum)
 * or 5, 7 (thermal).  c: Q*3 ints, w: Q (NULL for thermal), M: Q*Q row-major. */
int oracle_lattice(int kind, int *Q, int *c, double *w, double *M);

int oracle_max_threads(void);

/* Threads the following calls use (OpenMP); returns the previous count.  n < 1 is ignored. */
int oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
