/*
 * lbm_oracle.c -- plain, slow, fp64 CPU oracle of the lattice-Boltzmann collide-and-stream
 * step.  TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's
 * CPU-baseline leg; never by the product path.  It shares no code with the CUDA library.
 *
 * It follows the method as the pages state it, step by step, with two full buffers:
 *   "Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI", Sec. 2:
 *     Eq. 5 (MRT evolution of f with the forcing term F' = M^-1 (I - S/2) M F~),
 *     rho = sum f_i, u = (sum e_i f_i + F/2)/rho, F = rho g beta_T (T - T0) along the
 *     vertical unit vector, half-way bounce-back f_ibar(x, t+1) = f_i+(x, t),
 *     Eq. 7 (MRT evolution of g on D2Q5 / D3Q7), T = sum g_i, half-way anti-bounce-back
 *     g_ibar(x, t+1) = -g_i+(x, t) + omega T_w with omega = (4 + a_T)/10 (D2Q5) or
 *     (6 + a_T)/21 (D3Q7), and half-way bounce-back for adiabatic walls;
 *     Sec. 3 (SoA index x + Nx y + Nx Ny z + Nx Ny Nz i).
 *   "GPU Optimization for High-Quality Kinetic Fluid Simulation", Sec. 3.1: Eq. 1 (LBE),
 *     Eq. 2 (moments), Eq. 3 (pull streaming f*(x) = f(x - c_i)), Eq. 5 (MRT collision
 *     Omega = -M^-1 D (m - m_eq)); Fig. 6 / Alg. 1 (bounce-back at solid nodes).
 *   "GPU lattice Boltzmann: streaming layout and performance": the two-buffer scheme
 *     (collide, then pull into the other buffer) and momentum exchange on wall links.
 *
 * Where the pages are silent the oracle takes these readings (each also listed in the
 * design notes): d'Humieres D3Q19 moment basis and Lallemand-Luo D2Q9 basis with the
 * compressible quadratic equilibrium, m_eq = M f_eq; Guo's velocity-space source F~
 * mapped literally through M^-1 (I - S/2) M; rates of conserved moments are 0;
 * thermal equilibrium moments (T, u T, a_T T, 0...) for D2Q5/D3Q7; a link is a wall link
 * when its source lies outside the domain through a WALL face or is a solid cell; solid
 * links are adiabatic for g; the momentum exchange is the sum of 2 f_i+ c_i over links
 * from fluid cells into solid cells (domain faces excluded).
 *
 * D3Q27 central-moment MRT ("GPU Optimization for High-Quality Kinetic Fluid Simulation",
 * Sec. 3.1: the D3Q27 lattice of Fig. 2 and Omega = -M^-1 D (m - m_eq) of Eq. 5, where M is
 * a central-moment matrix; the adaptive rates of its refs. [1, 2] are not available, so the
 * rates are fixed inputs).  Readings: M(u) has the rows prod_a (c_a - u_a)^e_a for
 * e in {0,1,2}^3, except that the second-order normal rows are taken as xx - yy, xx - zz
 * (relaxed with the shear rate 1/tau, like xy, xz, yz) and xx + yy + zz (bulk rate); the
 * third- to sixth-order rows each take their order's rate; rows of order 0 and 1 are
 * conserved.  The equilibrium is the product form rho prod_a phi(c_a, u_a) with
 * phi(0, u) = 2/3 - u^2 and phi(+-1, u) = (1/3 + u^2 +- u)/2, whose central moments are those
 * of a Maxwellian, rho prod_a (1, 0, 1/3)[e_a].  The force enters as Guo's does on the other
 * lattices: the source is (F/rho) . d f_eq / du, mapped through M^-1 (I - D/2) M, with
 * u = (j + F/2)/rho.  M(u) f = m is inverted by Gaussian elimination.
 */
#include "lbm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QMAX 27

typedef struct {
    int Q;
    int c[QMAX][3];
    double w[QMAX];
    int opp[QMAX];
    double M[QMAX][QMAX];
    double Minv[QMAX][QMAX];
} lattice_t;

/* ---------------------------------------------------------------- velocity sets -- */

/* D3Q19 in d'Humieres' order: rest; +-x, +-y, +-z; then the xy, xz, yz edge links, each
 * group ordered (+,+), (-,+), (+,-), (-,-). */
static const int C_D3Q19[19][3] = {
    {0, 0, 0},
    {1, 0, 0}, {-1, 0, 0}, {0, 1, 0}, {0, -1, 0}, {0, 0, 1}, {0, 0, -1},
    {1, 1, 0}, {-1, 1, 0}, {1, -1, 0}, {-1, -1, 0},
    {1, 0, 1}, {-1, 0, 1}, {1, 0, -1}, {-1, 0, -1},
    {0, 1, 1}, {0, -1, 1}, {0, 1, -1}, {0, -1, -1}};

/* D2Q9: rest, +x, +y, -x, -y, (+,+), (-,+), (-,-), (+,-); with this order f2, f5, f6
 * cross the top face and f4, f7, f8 the bottom face, as the multi-GPU thermal page's
 * halo description (Sec. 3.1, Fig. 3(b)) requires. */
/* D3Q27: the D3Q19 order, then the corners (+,+,+), (-,+,+), (+,-,+), (-,-,+), (+,+,-),
 * (-,+,-), (+,-,-), (-,-,-). */
static const int C_D3Q27[27][3] = {
    {0, 0, 0},
    {1, 0, 0}, {-1, 0, 0}, {0, 1, 0}, {0, -1, 0}, {0, 0, 1}, {0, 0, -1},
    {1, 1, 0}, {-1, 1, 0}, {1, -1, 0}, {-1, -1, 0},
    {1, 0, 1}, {-1, 0, 1}, {1, 0, -1}, {-1, 0, -1},
    {0, 1, 1}, {0, -1, 1}, {0, 1, -1}, {0, -1, -1},
    {1, 1, 1}, {-1, 1, 1}, {1, -1, 1}, {-1, -1, 1},
    {1, 1, -1}, {-1, 1, -1}, {1, -1, -1}, {-1, -1, -1}};

static const int C_D2Q9[9][3] = {
    {0, 0, 0}, {1, 0, 0}, {0, 1, 0}, {-1, 0, 0}, {0, -1, 0},
    {1, 1, 0}, {-1, 1, 0}, {-1, -1, 0}, {1, -1, 0}};

/* D3Q7: rest, +x, -x, +y, -y, +z, -z.  D2Q5: rest, +x, +y, -x, -y. */
static const int C_D3Q7[7][3] = {
    {0, 0, 0}, {1, 0, 0}, {-1, 0, 0}, {0, 1, 0}, {0, -1, 0}, {0, 0, 1}, {0, 0, -1}};
static const int C_D2Q5[5][3] = {{0, 0, 0}, {1, 0, 0}, {0, 1, 0}, {-1, 0, 0}, {0, -1, 0}};

/* ----------------------------------------------------------------- moment bases -- */

/* d'Humieres et al. (2002) D3Q19 basis as polynomials of c (c2 = |c|^2):
 * rho, e, eps, jx, qx, jy, qy, jz, qz, 3pxx, 3pixx, pww, piww, pxy, pyz, pxz, mx, my, mz */
static double row_d3q19(int k, const int *c)
{
    const double cx = c[0], cy = c[1], cz = c[2];
    const double c2 = cx * cx + cy * cy + cz * cz;
    switch (k) {
    case 0: return 1.0;
    case 1: return 19.0 * c2 - 30.0;
    case 2: return (21.0 * c2 * c2 - 53.0 * c2 + 24.0) / 2.0;
    case 3: return cx;
    case 4: return (5.0 * c2 - 9.0) * cx;
    case 5: return cy;
    case 6: return (5.0 * c2 - 9.0) * cy;
    case 7: return cz;
    case 8: return (5.0 * c2 - 9.0) * cz;
    case 9: return 3.0 * cx * cx - c2;
    case 10: return (3.0 * c2 - 5.0) * (3.0 * cx * cx - c2);
    case 11: return cy * cy - cz * cz;
    case 12: return (3.0 * c2 - 5.0) * (cy * cy - cz * cz);
    case 13: return cx * cy;
    case 14: return cy * cz;
    case 15: return cx * cz;
    case 16: return (cy * cy - cz * cz) * cx;
    case 17: return (cz * cz - cx * cx) * cy;
    default: return (cx * cx - cy * cy) * cz;
    }
}

/* Lallemand-Luo (2000) D2Q9 basis: rho, e, eps, jx, qx, jy, qy, pxx, pxy */
static double row_d2q9(int k, const int *c)
{
    const double cx = c[0], cy = c[1];
    const double c2 = cx * cx + cy * cy;
    switch (k) {
    case 0: return 1.0;
    case 1: return 3.0 * c2 - 4.0;
    case 2: return (9.0 * c2 * c2 - 21.0 * c2 + 8.0) / 2.0;
    case 3: return cx;
    case 4: return (3.0 * c2 - 5.0) * cx;
    case 5: return cy;
    case 6: return (3.0 * c2 - 5.0) * cy;
    case 7: return cx * cx - cy * cy;
    default: return cx * cy;
    }
}

/* Thermal bases: T, jx, jy, (jz), energy (rest weight -(Q-1)), anisotropic rows. */
static const double N_D3Q7[7][7] = {
    {1, 1, 1, 1, 1, 1, 1},
    {0, 1, -1, 0, 0, 0, 0},
    {0, 0, 0, 1, -1, 0, 0},
    {0, 0, 0, 0, 0, 1, -1},
    {-6, 1, 1, 1, 1, 1, 1},
    {0, 2, 2, -1, -1, -1, -1},
    {0, 0, 0, 1, 1, -1, -1}};
static const double N_D2Q5[5][5] = {
    {1, 1, 1, 1, 1},
    {0, 1, 0, -1, 0},
    {0, 0, 1, 0, -1},
    {-4, 1, 1, 1, 1},
    {0, 1, -1, 1, -1}};

/* Fill a lattice: velocities, weights (momentum lattices), opposites, M and
 * M^-1 = M^T diag(1/|row|^2), after checking that the rows are mutually orthogonal. */
static int make_lattice(int kind, lattice_t *L)
{
    memset(L, 0, sizeof(*L));
    const int(*c)[3];
    switch (kind) {
    case 19: L->Q = 19; c = C_D3Q19; break;
    case 27: L->Q = 27; c = C_D3Q27; break;
    case 9: L->Q = 9; c = C_D2Q9; break;
    case 7: L->Q = 7; c = C_D3Q7; break;
    case 5: L->Q = 5; c = C_D2Q5; break;
    default: return -1;
    }
    const int Q = L->Q;
    for (int q = 0; q < Q; ++q)
        for (int a = 0; a < 3; ++a) L->c[q][a] = c[q][a];
    for (int q = 0; q < Q; ++q) {
        L->opp[q] = -1;
        for (int p = 0; p < Q; ++p)
            if (c[p][0] == -c[q][0] && c[p][1] == -c[q][1] && c[p][2] == -c[q][2]) L->opp[q] = p;
        if (L->opp[q] < 0) return -2;
    }
    for (int q = 0; q < Q; ++q) {
        const int c2 = c[q][0] * c[q][0] + c[q][1] * c[q][1] + c[q][2] * c[q][2];
        if (kind == 19) L->w[q] = (c2 == 0) ? 1.0 / 3.0 : (c2 == 1) ? 1.0 / 18.0 : 1.0 / 36.0;
        if (kind == 9) L->w[q] = (c2 == 0) ? 4.0 / 9.0 : (c2 == 1) ? 1.0 / 9.0 : 1.0 / 36.0;
        /* D3Q27: product of the D1Q3 weights 2/3 (rest) and 1/6 (moving) */
        if (kind == 27)
            L->w[q] = (c2 == 0) ? 8.0 / 27.0 : (c2 == 1) ? 2.0 / 27.0 : (c2 == 2) ? 1.0 / 54.0
                                                                             : 1.0 / 216.0;
    }
    if (kind == 27) return 0;   /* the central-moment matrix depends on u: built per cell */
    for (int k = 0; k < Q; ++k)
        for (int q = 0; q < Q; ++q) {
            if (kind == 19) L->M[k][q] = row_d3q19(k, c[q]);
            else if (kind == 9) L->M[k][q] = row_d2q9(k, c[q]);
            else if (kind == 7) L->M[k][q] = N_D3Q7[k][q];
            else L->M[k][q] = N_D2Q5[k][q];
        }
    for (int a = 0; a < Q; ++a)
        for (int b = 0; b < Q; ++b) {
            double dot = 0.0;
            for (int q = 0; q < Q; ++q) dot += L->M[a][q] * L->M[b][q];
            if (a != b && dot != 0.0) return -3;
            if (a == b) {
                if (dot <= 0.0) return -3;
                for (int q = 0; q < Q; ++q) L->Minv[q][a] = L->M[a][q] / dot;
            }
        }
    return 0;
}

/* ------------------------------------------------------------------- the problem -- */

typedef struct {
    const oracle_problem *p;
    lattice_t F;     /* momentum lattice */
    lattice_t G;     /* thermal lattice (Q = 0 if none) */
    double s[QMAX];  /* rates per moment row, conserved rows zeroed */
    double sT[7];
    double omega;    /* anti-bounce-back weight */
    long W;
} ctx_t;

/* Exponents (e_x, e_y, e_z) of the D3Q27 central-moment rows.  Rows 7, 8, 9 are the
 * recombined second-order normal moments xx - yy, xx - zz, xx + yy + zz (see cm_row). */
static const int CM_EXP[27][3] = {
    {0, 0, 0},
    {1, 0, 0}, {0, 1, 0}, {0, 0, 1},
    {1, 1, 0}, {1, 0, 1}, {0, 1, 1},
    {2, 0, 0}, {0, 2, 0}, {0, 0, 2},
    {1, 2, 0}, {1, 0, 2}, {2, 1, 0}, {0, 1, 2}, {2, 0, 1}, {0, 2, 1}, {1, 1, 1},
    {2, 2, 0}, {2, 0, 2}, {0, 2, 2}, {2, 1, 1}, {1, 2, 1}, {1, 1, 2},
    {2, 2, 1}, {2, 1, 2}, {1, 2, 2},
    {2, 2, 2}};

/* Rate of D3Q27 central-moment row k: 0 for the conserved orders 0 and 1, the shear rate
 * for xy, xz, yz, xx - yy, xx - zz, the bulk rate for xx + yy + zz, then one rate per
 * order (rows 10-16: third, 17-22: fourth, 23-25: fifth, 26: sixth). */
static double cm_rate(const oracle_problem *p, int k)
{
    if (k < 4) return 0.0;
    if (k < 9) return 1.0 / p->tau;
    if (k == 9) return p->cm_rates[0];
    if (k < 17) return p->cm_rates[1];
    if (k < 23) return p->cm_rates[2];
    if (k < 26) return p->cm_rates[3];
    return p->cm_rates[4];
}

static int is_conserved_row(int lattice, int k)
{
    if (lattice == 27) return k < 4;
    if (lattice == 19) return k == 0 || k == 3 || k == 5 || k == 7;
    return k == 0 || k == 3 || k == 5;
}

int oracle_check(const oracle_problem *p)
{
    if (!p) return -1;
    if (p->lattice != 19 && p->lattice != 9 && p->lattice != 27) return -2;
    if (p->thermal != 0 && !((p->lattice == 19 && p->thermal == 7) ||
                             (p->lattice == 9 && p->thermal == 5)))
        return -3;
    if (p->lattice == 27 ? p->collision != ORC_CM
                         : (p->collision != ORC_BGK && p->collision != ORC_MRT))
        return -4;
    if (p->lattice == 27) {
        if (!(p->tau > 0.5)) return -9;
        for (int k = 0; k < 5; ++k)
            if (!(p->cm_rates[k] > 0.0 && p->cm_rates[k] < 2.0)) return -13;
    }
    if (p->nx < 1 || p->ny < 1 || p->nz < 1) return -5;
    if (p->lattice == 9 && p->nz != 1) return -6;
    if (p->wx < 1 || p->wy < 1 || p->wz < 1) return -7;
    if (p->x0 < 0 || p->y0 < 0 || p->z0 < 0 || p->x0 + p->wx > p->nx ||
        p->y0 + p->wy > p->ny || p->z0 + p->wz > p->nz)
        return -8;
    if (p->collision == ORC_BGK && !(p->tau > 0.5)) return -9;
    if (p->up_axis < 0 || p->up_axis > 2) return -10;
    if (p->ib_n < 0 || (p->ib_n > 0 && !p->ib_x)) return -12;
    for (int i = 0; i < 6; ++i)
        if ((p->face_flow[i] != ORC_PERIODIC && p->face_flow[i] != ORC_WALL) ||
            (p->face_T[i] != ORC_ADIABATIC && p->face_T[i] != ORC_DIRICHLET))
            return -11;
    return 0;
}

static int make_ctx(const oracle_problem *p, ctx_t *C)
{
    int rc = oracle_check(p);
    if (rc) return rc;
    memset(C, 0, sizeof(*C));
    C->p = p;
    if (make_lattice(p->lattice, &C->F)) return -20;
    if (p->thermal && make_lattice(p->thermal, &C->G)) return -21;
    for (int k = 0; k < C->F.Q; ++k)
        C->s[k] = is_conserved_row(p->lattice, k) ? 0.0
                  : (p->lattice == 27)           ? cm_rate(p, k)
                                                 : p->s[k];
    for (int k = 0; k < C->G.Q; ++k) C->sT[k] = (k == 0) ? 0.0 : p->s_T[k];
    /* anti-bounce-back weight as the thermal page prints it */
    if (p->thermal == 5) C->omega = (4.0 + p->a_T) / 10.0;
    if (p->thermal == 7) C->omega = (6.0 + p->a_T) / 21.0;
    C->W = (long)p->wx * p->wy * p->wz;
    return 0;
}

static int is_solid(const ctx_t *C, long n) { return C->p->solid && C->p->solid[n]; }

/* ------------------------------------------------------------- per-cell physics -- */

/* Body force per the thermal page: F = rho g_body + rho g beta (T - T0) e_up. */
static void body_force(const ctx_t *C, double rho, double T, double F[3])
{
    const oracle_problem *p = C->p;
    for (int a = 0; a < 3; ++a) F[a] = rho * p->g_body[a];
    if (p->thermal) F[p->up_axis] += rho * p->gbeta * (T - p->T0);
}

/* D1Q3 factor of the D3Q27 product equilibrium: its zeroth, first and second moments are
 * 1, u and 1/3 + u^2, those of a Maxwellian with c_s^2 = 1/3. */
static double phi(int c, double u)
{
    return c == 0 ? 2.0 / 3.0 - u * u : 0.5 * (1.0 / 3.0 + u * u + c * u);
}

/* d phi / du */
static double dphi(int c, double u) { return c == 0 ? -2.0 * u : u + 0.5 * c; }

/* Equilibrium.  D3Q27: the product form rho prod_a phi(c_a, u_a).  Otherwise the quadratic
 * f_eq_q = w_q rho (1 + 3 c.u + 9/2 (c.u)^2 - 3/2 u.u). */
static void f_equilibrium(const lattice_t *L, double rho, const double u[3], double *feq)
{
    if (L->Q == 27) {
        for (int q = 0; q < 27; ++q)
            feq[q] = rho * phi(L->c[q][0], u[0]) * phi(L->c[q][1], u[1]) * phi(L->c[q][2], u[2]);
        return;
    }
    const double uu = u[0] * u[0] + u[1] * u[1] + u[2] * u[2];
    for (int q = 0; q < L->Q; ++q) {
        const double cu = L->c[q][0] * u[0] + L->c[q][1] * u[1] + L->c[q][2] * u[2];
        feq[q] = L->w[q] * rho * (1.0 + 3.0 * cu + 4.5 * cu * cu - 1.5 * uu);
    }
}

/* Thermal equilibrium moments on the D2Q5 / D3Q7 bases: T, u T, a_T T, then zeros. */
static void g_equilibrium_moments(const ctx_t *C, double T, const double u[3], double *neq)
{
    const int dim = (C->G.Q == 7) ? 3 : 2;
    for (int k = 0; k < C->G.Q; ++k) neq[k] = 0.0;
    neq[0] = T;
    for (int a = 0; a < dim; ++a) neq[1 + a] = u[a] * T;
    neq[1 + dim] = C->p->a_T * T;
}

/* g_eq = N^-1 n_eq */
static void g_equilibrium(const ctx_t *C, double T, const double u[3], double *geq)
{
    const lattice_t *G = &C->G;
    double neq[7];
    g_equilibrium_moments(C, T, u, neq);
    for (int q = 0; q < G->Q; ++q) {
        double v = 0.0;
        for (int k = 0; k < G->Q; ++k) v += G->Minv[q][k] * neq[k];
        geq[q] = v;
    }
}

/* Guo's source in velocity space: F~_q = w_q [3 (c_q - u) + 9 (c_q.u) c_q] . F, which is
 * (F/rho) . d f_eq / du of the quadratic equilibrium.  D3Q27: (F/rho) . d f_eq / du of the
 * product form. */
static void guo_source(const lattice_t *L, const double u[3], const double F[3], double *Ft)
{
    if (L->Q == 27) {
        for (int q = 0; q < 27; ++q) {
            const int *c = L->c[q];
            const double px = phi(c[0], u[0]), py = phi(c[1], u[1]), pz = phi(c[2], u[2]);
            Ft[q] = F[0] * dphi(c[0], u[0]) * py * pz + F[1] * px * dphi(c[1], u[1]) * pz +
                    F[2] * px * py * dphi(c[2], u[2]);
        }
        return;
    }
    for (int q = 0; q < L->Q; ++q) {
        const double cu = L->c[q][0] * u[0] + L->c[q][1] * u[1] + L->c[q][2] * u[2];
        double v = 0.0;
        for (int a = 0; a < 3; ++a) v += (3.0 * (L->c[q][a] - u[a]) + 9.0 * cu * L->c[q][a]) * F[a];
        Ft[q] = L->w[q] * v;
    }
}

/* Central moment of velocity c about u with exponents e: prod_a (c_a - u_a)^e_a. */
static double cmono(const int *c, const double u[3], const int *e)
{
    double v = 1.0;
    for (int a = 0; a < 3; ++a)
        for (int n = 0; n < e[a]; ++n) v *= c[a] - u[a];
    return v;
}

/* Entry (k, c) of the central-moment matrix M(u). */
static double cm_row(int k, const int *c, const double u[3])
{
    static const int XX[3] = {2, 0, 0}, YY[3] = {0, 2, 0}, ZZ[3] = {0, 0, 2};
    if (k == 7) return cmono(c, u, XX) - cmono(c, u, YY);
    if (k == 8) return cmono(c, u, XX) - cmono(c, u, ZZ);
    if (k == 9) return cmono(c, u, XX) + cmono(c, u, YY) + cmono(c, u, ZZ);
    return cmono(c, u, CM_EXP[k]);
}

/* Solve A x = b for n <= QMAX by Gaussian elimination with partial pivoting (A and b are
 * overwritten).  Returns -1 on a singular matrix. */
static int solve_dense(int n, double A[][QMAX], double *b, double *x)
{
    for (int col = 0; col < n; ++col) {
        int piv = col;
        for (int r = col + 1; r < n; ++r)
            if (fabs(A[r][col]) > fabs(A[piv][col])) piv = r;
        if (A[piv][col] == 0.0) return -1;
        if (piv != col) {
            for (int k = 0; k < n; ++k) {
                const double t = A[col][k];
                A[col][k] = A[piv][k];
                A[piv][k] = t;
            }
            const double t = b[col];
            b[col] = b[piv];
            b[piv] = t;
        }
        for (int r = col + 1; r < n; ++r) {
            const double m = A[r][col] / A[col][col];
            if (m == 0.0) continue;
            for (int k = col; k < n; ++k) A[r][k] -= m * A[col][k];
            b[r] -= m * b[col];
        }
    }
    for (int r = n - 1; r >= 0; --r) {
        double v = b[r];
        for (int k = r + 1; k < n; ++k) v -= A[r][k] * x[k];
        x[r] = v / A[r][r];
    }
    return 0;
}

/* Collide one fluid cell: fin/gin -> fout/gout (post-collision).  Fext: additional force
 * on the cell (the immersed boundary's), added to the body force. */
static void collide_cell(const ctx_t *C, const double *fin, const double *gin, double *fout,
                         double *gout, const double *Fext)
{
    const lattice_t *L = &C->F;
    const int Q = L->Q;
    /* moments */
    double rho = 0.0, j[3] = {0, 0, 0}, T = 0.0;
    for (int q = 0; q < Q; ++q) {
        rho += fin[q];
        for (int a = 0; a < 3; ++a) j[a] += L->c[q][a] * fin[q];
    }
    if (C->p->thermal)
        for (int k = 0; k < C->G.Q; ++k) T += gin[k];
    /* force and velocity */
    double F[3], u[3];
    body_force(C, rho, T, F);
    for (int a = 0; a < 3; ++a) F[a] += Fext[a];
    for (int a = 0; a < 3; ++a) u[a] = (j[a] + 0.5 * F[a]) / rho;
    /* equilibrium and source */
    double feq[QMAX], Ft[QMAX];
    f_equilibrium(L, rho, u, feq);
    guo_source(L, u, F, Ft);
    if (C->p->collision == ORC_CM) {
        /* m = M(u) f, relax each row toward m_eq = M(u) f_eq with its rate, add
         * (I - D/2) M(u) F~, and solve M(u) f_out = m_post */
        double A[QMAX][QMAX], m[QMAX], meq[QMAX], mF[QMAX], mpost[QMAX];
        for (int k = 0; k < Q; ++k) {
            double a = 0.0, b = 0.0, d = 0.0;
            for (int q = 0; q < Q; ++q) {
                A[k][q] = cm_row(k, L->c[q], u);
                a += A[k][q] * fin[q];
                b += A[k][q] * feq[q];
                d += A[k][q] * Ft[q];
            }
            m[k] = a;
            meq[k] = b;
            mF[k] = d;
        }
        for (int k = 0; k < Q; ++k)
            mpost[k] = m[k] - C->s[k] * (m[k] - meq[k]) + (1.0 - 0.5 * C->s[k]) * mF[k];
        if (solve_dense(Q, A, mpost, fout))
            for (int q = 0; q < Q; ++q) fout[q] = NAN;
    } else if (C->p->collision == ORC_BGK) {
        const double tau = C->p->tau;
        for (int q = 0; q < Q; ++q)
            fout[q] = fin[q] - (fin[q] - feq[q]) / tau + (1.0 - 1.0 / (2.0 * tau)) * Ft[q];
    } else {
        double m[QMAX], meq[QMAX], mF[QMAX], mpost[QMAX];
        for (int k = 0; k < Q; ++k) {
            double a = 0.0, b = 0.0, d = 0.0;
            for (int q = 0; q < Q; ++q) {
                a += L->M[k][q] * fin[q];
                b += L->M[k][q] * feq[q];
                d += L->M[k][q] * Ft[q];
            }
            m[k] = a;
            meq[k] = b;
            mF[k] = d;
        }
        for (int k = 0; k < Q; ++k)
            mpost[k] = m[k] - C->s[k] * (m[k] - meq[k]) + (1.0 - 0.5 * C->s[k]) * mF[k];
        for (int q = 0; q < Q; ++q) {
            double v = 0.0;
            for (int k = 0; k < Q; ++k) v += L->Minv[q][k] * mpost[k];
            fout[q] = v;
        }
    }
    if (C->p->thermal) {
        const lattice_t *G = &C->G;
        double n[7], neq[7], npost[7];
        g_equilibrium_moments(C, T, u, neq);
        for (int k = 0; k < G->Q; ++k) {
            double a = 0.0;
            for (int q = 0; q < G->Q; ++q) a += G->M[k][q] * gin[q];
            n[k] = a;
        }
        for (int k = 0; k < G->Q; ++k) npost[k] = n[k] - C->sT[k] * (n[k] - neq[k]);
        for (int q = 0; q < G->Q; ++q) {
            double v = 0.0;
            for (int k = 0; k < G->Q; ++k) v += G->Minv[q][k] * npost[k];
            gout[q] = v;
        }
    }
}

/* ------------------------------------------------------------------- streaming -- */

enum { SRC_CELL = 0, SRC_FACE_WALL = 1, SRC_SOLID = 2, SRC_UNKNOWN = 3 };

/* Classify the pull source x - c of window cell (i, j, k).  On SRC_CELL, *n_src is its
 * window index; on SRC_FACE_WALL, *face is the face the link leaves through. */
static int pull_source(const ctx_t *C, int i, int j, int k, const int *c, long *n_src, int *face)
{
    const oracle_problem *p = C->p;
    const int ext[3] = {p->nx, p->ny, p->nz};
    const int org[3] = {p->x0, p->y0, p->z0};
    const int win[3] = {p->wx, p->wy, p->wz};
    int s[3] = {p->x0 + i - c[0], p->y0 + j - c[1], p->z0 + k - c[2]};
    int wall_face = -1;
    for (int a = 0; a < 3; ++a) {
        if (s[a] < 0) {
            if (p->face_flow[2 * a] == ORC_WALL) wall_face = 2 * a;
            else s[a] += ext[a];
        } else if (s[a] >= ext[a]) {
            if (p->face_flow[2 * a + 1] == ORC_WALL) wall_face = 2 * a + 1;
            else s[a] -= ext[a];
        }
    }
    if (wall_face >= 0) {
        *face = wall_face;
        return SRC_FACE_WALL;
    }
    for (int a = 0; a < 3; ++a) {
        s[a] -= org[a];
        if (s[a] < 0 || s[a] >= win[a]) return SRC_UNKNOWN;
    }
    *n_src = s[0] + (long)p->wx * (s[1] + (long)p->wy * s[2]);
    return is_solid(C, *n_src) ? SRC_SOLID : SRC_CELL;
}

/* ------------------------------------------------------------ immersed boundary -- */

/* Window index of the stencil node base + d (d in {0,1}^3) of a sample, or -1 if it is
 * outside the window (unknown), -2 if it leaves the domain through a wall face. */
static long stencil_node(const ctx_t *C, const int base[3], const int d[3])
{
    const oracle_problem *p = C->p;
    const int ext[3] = {p->nx, p->ny, p->nz};
    const int org[3] = {p->x0, p->y0, p->z0};
    const int win[3] = {p->wx, p->wy, p->wz};
    int s[3];
    for (int a = 0; a < 3; ++a) {
        s[a] = base[a] + d[a];
        if (s[a] < 0 || s[a] >= ext[a]) {
            if (p->face_flow[2 * a + (s[a] >= ext[a])] == ORC_WALL) return -2;
            s[a] = (s[a] % ext[a] + ext[a]) % ext[a];
        }
        s[a] -= org[a];
        if (s[a] < 0 || s[a] >= win[a]) return -1;
    }
    return s[0] + (long)p->wx * (s[1] + (long)p->wy * s[2]);
}

/* Immersed-boundary force per cell (Fib, 3 planes of W), from the state f, g at time t:
 * interpolate rho and u = (j + F_body/2)/rho to each sample with the trilinear kernel
 * (Eq. 6), penalty g_s = w rho (u_b - u) (Eq. 7), spread with the same kernel (Eq. 8).
 * Solid cells contribute rho = 1, u = 0 and receive nothing.  Unknown stencil nodes make
 * the sample's force NaN.  ib[6] gets -sum g_s and -sum (x_s - centroid) x g_s. */
static int ib_forces(const ctx_t *C, const double *f, const double *g, double *Fib, double ib[6])
{
    const oracle_problem *p = C->p;
    const long W = C->W;
    const int dim = (p->lattice != 9) ? 3 : 2;
    for (long n = 0; n < 3 * W; ++n) Fib[n] = 0.0;
    double total[3] = {0, 0, 0}, torque[3] = {0, 0, 0}, centre[3] = {0, 0, 0};
    for (int s = 0; s < p->ib_n; ++s)
        for (int a = 0; a < 3; ++a) centre[a] += p->ib_x[3 * s + a] / p->ib_n;
    for (int s = 0; s < p->ib_n; ++s) {
        const double *xs = p->ib_x + 3 * s;
        int base[3] = {0, 0, 0};
        double fr[3] = {0, 0, 0};
        for (int a = 0; a < dim; ++a) {
            base[a] = (int)floor(xs[a]);
            fr[a] = xs[a] - base[a];
        }
        long node[8];
        double K[8];
        int nn = 0;
        double rho = 0.0, u[3] = {0, 0, 0};
        for (int dz = 0; dz <= (dim == 3); ++dz)
            for (int dy = 0; dy <= 1; ++dy)
                for (int dx = 0; dx <= 1; ++dx) {
                    const int d[3] = {dx, dy, dz};
                    double k = 1.0;
                    for (int a = 0; a < dim; ++a) k *= d[a] ? fr[a] : 1.0 - fr[a];
                    const long nidx = stencil_node(C, base, d);
                    if (nidx == -2) return -60;
                    node[nn] = nidx;
                    K[nn++] = k;
                    if (nidx < 0) {
                        rho = NAN;
                        continue;
                    }
                    double r = 1.0, v[3] = {0, 0, 0};
                    if (!is_solid(C, nidx)) {
                        double j[3] = {0, 0, 0}, T = 0.0, F[3];
                        r = 0.0;
                        for (int q = 0; q < C->F.Q; ++q) {
                            r += f[q * W + nidx];
                            for (int a = 0; a < 3; ++a) j[a] += C->F.c[q][a] * f[q * W + nidx];
                        }
                        for (int q = 0; q < C->G.Q; ++q) T += g[q * W + nidx];
                        body_force(C, r, T, F);
                        for (int a = 0; a < 3; ++a) v[a] = (j[a] + 0.5 * F[a]) / r;
                    }
                    rho += k * r;
                    for (int a = 0; a < 3; ++a) u[a] += k * v[a];
                }
        const double w = p->ib_w ? p->ib_w[s] : 1.0;
        double gs[3];
        for (int a = 0; a < 3; ++a) {
            const double ub = p->ib_ub ? p->ib_ub[3 * s + a] : 0.0;
            gs[a] = (a < dim) ? w * rho * (ub - u[a]) : 0.0;
            total[a] -= gs[a];
        }
        const double r[3] = {xs[0] - centre[0], xs[1] - centre[1], xs[2] - centre[2]};
        torque[0] -= r[1] * gs[2] - r[2] * gs[1];
        torque[1] -= r[2] * gs[0] - r[0] * gs[2];
        torque[2] -= r[0] * gs[1] - r[1] * gs[0];
        for (int i = 0; i < nn; ++i) {
            if (node[i] < 0 || is_solid(C, node[i])) continue;
            for (int a = 0; a < 3; ++a) Fib[a * W + node[i]] += K[i] * gs[a];
        }
    }
    if (ib) {
        for (int a = 0; a < 3; ++a) {
            ib[a] = total[a];
            ib[3 + a] = torque[a];
        }
    }
    return 0;
}

/* --------------------------------------------------------------------- the API -- */

int oracle_init_equilibrium(const oracle_problem *p, const double *rho, const double *u,
                            const double *T, double *f, double *g)
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    if (p->thermal && !T) return -30;
    const long W = C.W;
#pragma omp parallel for schedule(static)
    for (long n = 0; n < W; ++n) {
        double feq[QMAX], geq[7];
        if (is_solid(&C, n)) {
            for (int q = 0; q < C.F.Q; ++q) f[q * W + n] = 0.0;
            for (int q = 0; q < C.G.Q; ++q) g[q * W + n] = 0.0;
            continue;
        }
        const double un[3] = {u[n], u[W + n], (p->lattice != 9) ? u[2 * W + n] : 0.0};
        f_equilibrium(&C.F, rho[n], un, feq);
        for (int q = 0; q < C.F.Q; ++q) f[q * W + n] = feq[q];
        if (p->thermal) {
            g_equilibrium(&C, T[n], un, geq);
            for (int q = 0; q < C.G.Q; ++q) g[q * W + n] = geq[q];
        }
    }
    return 0;
}

int oracle_step(const oracle_problem *p, double *f, double *g, double *fpost, double *gpost,
                double force[3], double ib[6])
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    const long W = C.W;
    const int Q = C.F.Q, QT = C.G.Q;
    const int wx = p->wx, wy = p->wy, wz = p->wz;

    /* 0. immersed-boundary force of this step, from the state at t */
    double *Fib = NULL;
    if (p->ib_n > 0) {
        Fib = (double *)malloc(sizeof(double) * 3 * (size_t)W);
        if (!Fib) return -40;
        rc = ib_forces(&C, f, g, Fib, ib);
        if (rc) {
            free(Fib);
            return rc;
        }
    } else if (ib) {
        for (int a = 0; a < 6; ++a) ib[a] = 0.0;
    }

    /* 1. collide every fluid cell into the second buffer; solid cells hold NaN there so
     *    that a read of them would show up in the results. */
#pragma omp parallel for schedule(static)
    for (long n = 0; n < W; ++n) {
        double fin[QMAX], gin[7], fo[QMAX], go[7];
        if (is_solid(&C, n)) {
            for (int q = 0; q < Q; ++q) fpost[q * W + n] = NAN;
            for (int q = 0; q < QT; ++q) gpost[q * W + n] = NAN;
            continue;
        }
        for (int q = 0; q < Q; ++q) fin[q] = f[q * W + n];
        for (int q = 0; q < QT; ++q) gin[q] = g[q * W + n];
        const double Fext[3] = {Fib ? Fib[n] : 0.0, Fib ? Fib[W + n] : 0.0,
                                Fib ? Fib[2 * W + n] : 0.0};
        collide_cell(&C, fin, gin, fo, go, Fext);
        for (int q = 0; q < Q; ++q) fpost[q * W + n] = fo[q];
        for (int q = 0; q < QT; ++q) gpost[q * W + n] = go[q];
    }

    /* 2. pull streaming back into the state buffer, one x-row per task; the momentum
     *    exchange of each row is summed in row order afterwards. */
    const long rows = (long)wy * wz;
    double *row_force = (double *)calloc((size_t)rows * 3, sizeof(double));
    if (!row_force) {
        free(Fib);
        return -40;
    }
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const int j = (int)(r % wy), k = (int)(r / wy);
        double pf[3] = {0, 0, 0};
        for (int i = 0; i < wx; ++i) {
            const long n = i + (long)wx * (j + (long)wy * k);
            if (is_solid(&C, n)) {
                for (int q = 0; q < Q; ++q) f[q * W + n] = 0.0;
                for (int q = 0; q < QT; ++q) g[q * W + n] = 0.0;
                continue;
            }
            for (int q = 0; q < Q; ++q) {
                long ns = 0;
                int face = -1;
                const int kind = pull_source(&C, i, j, k, C.F.c[q], &ns, &face);
                const int o = C.F.opp[q];
                if (kind == SRC_CELL) {
                    f[q * W + n] = fpost[q * W + ns];
                } else if (kind == SRC_UNKNOWN) {
                    f[q * W + n] = NAN;
                } else {
                    /* half-way bounce-back: f_q(x, t+1) = f+_opp(q)(x, t) */
                    const double v = fpost[o * W + n];
                    f[q * W + n] = v;
                    if (kind == SRC_SOLID)
                        for (int a = 0; a < 3; ++a) pf[a] += 2.0 * v * C.F.c[o][a];
                }
            }
            for (int q = 0; q < QT; ++q) {
                long ns = 0;
                int face = -1;
                const int kind = pull_source(&C, i, j, k, C.G.c[q], &ns, &face);
                const int o = C.G.opp[q];
                if (kind == SRC_CELL) {
                    g[q * W + n] = gpost[q * W + ns];
                } else if (kind == SRC_UNKNOWN) {
                    g[q * W + n] = NAN;
                } else if (kind == SRC_FACE_WALL && p->face_T[face] == ORC_DIRICHLET) {
                    /* half-way anti-bounce-back: g_q = -g+_opp(q) + omega T_w */
                    g[q * W + n] = -gpost[o * W + n] + C.omega * p->T_wall[face];
                } else {
                    /* adiabatic wall or solid: half-way bounce-back */
                    g[q * W + n] = gpost[o * W + n];
                }
            }
        }
        row_force[3 * r + 0] = pf[0];
        row_force[3 * r + 1] = pf[1];
        row_force[3 * r + 2] = pf[2];
    }
    if (force) {
        force[0] = force[1] = force[2] = 0.0;
        for (long r = 0; r < rows; ++r)
            for (int a = 0; a < 3; ++a) force[a] += row_force[3 * r + a];
    }
    free(row_force);
    free(Fib);
    return 0;
}

int oracle_run(const oracle_problem *p, double *f, double *g, int steps, double force[3],
               double ib[6])
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    if (steps < 0) return -50;
    double *fpost = (double *)malloc(sizeof(double) * (size_t)C.W * C.F.Q);
    double *gpost = (double *)malloc(sizeof(double) * (size_t)C.W * (C.G.Q ? C.G.Q : 1));
    if (!fpost || !gpost) {
        free(fpost);
        free(gpost);
        return -40;
    }
    if (force) force[0] = force[1] = force[2] = 0.0;
    if (ib)
        for (int a = 0; a < 6; ++a) ib[a] = 0.0;
    for (int t = 0; t < steps && rc == 0; ++t) rc = oracle_step(p, f, g, fpost, gpost, force, ib);
    free(fpost);
    free(gpost);
    return rc;
}

int oracle_macroscopic(const oracle_problem *p, const double *f, const double *g, double *rho,
                       double *u, double *T)
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    const long W = C.W;
    const int dim = (p->lattice != 9) ? 3 : 2;
#pragma omp parallel for schedule(static)
    for (long n = 0; n < W; ++n) {
        if (is_solid(&C, n)) {
            rho[n] = 0.0;
            for (int a = 0; a < dim; ++a) u[a * W + n] = 0.0;
            if (T) T[n] = 0.0;
            continue;
        }
        double r = 0.0, j[3] = {0, 0, 0}, t = 0.0, F[3];
        for (int q = 0; q < C.F.Q; ++q) {
            r += f[q * W + n];
            for (int a = 0; a < 3; ++a) j[a] += C.F.c[q][a] * f[q * W + n];
        }
        for (int q = 0; q < C.G.Q; ++q) t += g[q * W + n];
        body_force(&C, r, t, F);
        rho[n] = r;
        for (int a = 0; a < dim; ++a) u[a * W + n] = (j[a] + 0.5 * F[a]) / r;
        if (T) T[n] = t;
    }
    return 0;
}

int oracle_diagnostics(const oracle_problem *p, const double *f, const double *g,
                       double out[13])
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    const long W = C.W;
    for (int i = 0; i < 13; ++i) out[i] = 0.0;
    for (int k = 0; k < p->wz; ++k)
        for (int j = 0; j < p->wy; ++j)
            for (int i = 0; i < p->wx; ++i) {
                const long n = i + (long)p->wx * (j + (long)p->wy * k);
                if (is_solid(&C, n)) continue;
                double t = 0.0, r = 0.0, jm[3] = {0, 0, 0};
                for (int q = 0; q < C.F.Q; ++q) {
                    out[0] += f[q * W + n];
                    r += f[q * W + n];
                    for (int a = 0; a < 3; ++a) {
                        out[1 + a] += C.F.c[q][a] * f[q * W + n];
                        jm[a] += C.F.c[q][a] * f[q * W + n];
                    }
                }
                for (int q = 0; q < C.G.Q; ++q) t += g[q * W + n];
                if (!p->thermal) continue;
                /* convective transport u T, u = (j + F/2)/rho as in the macroscopic fields */
                double F[3];
                body_force(&C, r, t, F);
                for (int a = 0; a < 3; ++a) out[10 + a] += (jm[a] + 0.5 * F[a]) / r * t;
                /* cells next to a Dirichlet face: wall gradient over the half cell */
                const int gc[3] = {p->x0 + i, p->y0 + j, p->z0 + k};
                const int ext[3] = {p->nx, p->ny, p->nz};
                const int dim = (p->lattice != 9) ? 3 : 2;
                for (int a = 0; a < dim; ++a) {
                    const int lo = 2 * a, hi = 2 * a + 1;
                    if (gc[a] == 0 && p->face_flow[lo] == ORC_WALL && p->face_T[lo] == ORC_DIRICHLET)
                        out[4 + lo] += 2.0 * (p->T_wall[lo] - t);
                    if (gc[a] == ext[a] - 1 && p->face_flow[hi] == ORC_WALL &&
                        p->face_T[hi] == ORC_DIRICHLET)
                        out[4 + hi] += 2.0 * (p->T_wall[hi] - t);
                }
            }
    return 0;
}

int oracle_lattice(int kind, int *Q, int *c, double *w, double *M)
{
    lattice_t L;
    if (make_lattice(kind, &L)) return -1;
    *Q = L.Q;
    for (int q = 0; q < L.Q; ++q) {
        for (int a = 0; a < 3; ++a) c[3 * q + a] = L.c[q][a];
        if (w) w[q] = L.w[q];
    }
    for (int k = 0; k < L.Q; ++k)
        for (int q = 0; q < L.Q; ++q) M[k * L.Q + q] = L.M[k][q];
    return 0;
}

int oracle_ib_forces(const oracle_problem *p, const double *f, const double *g, double *Fib,
                     double ib[6])
{
    ctx_t C;
    int rc = make_ctx(p, &C);
    if (rc) return rc;
    return ib_forces(&C, f, g, Fib, ib);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_set_threads(int n)
{
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}
