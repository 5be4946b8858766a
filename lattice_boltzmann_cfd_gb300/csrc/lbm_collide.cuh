// Per-cell collision of the CUDA path, in registers, fp32.
//
// Populations are stored shifted by their rest weights, fbar_q = f_q - w_q, so that fp32
// carries the deviations from rest with full relative precision; rho = 1 + sum fbar and
// every moment is linear, so the rest part only shifts the equilibria of the energy
// moments (e, eps) by their rest values.
//
// The method ("Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI",
// Sec. 2, Eq. 5 and Eq. 7; "GPU Optimization for High-Quality Kinetic Fluid Simulation",
// Sec. 3.1, Eq. 2 and Eq. 5):
//   rho = sum f, j = sum c f, T = sum g, F = rho g_body + rho g beta (T - T0) e_up,
//   u = (j + F/2) / rho,
//   MRT:  f+ = f + M^-1 [ -S (m - m_eq) + (I - S/2) M F~ ],  m = M f,
//   BGK:  f+ = f - (f - f_eq)/tau + (1 - 1/(2 tau)) F~,
//   g+ = g + N^-1 [ -S_T (n - n_eq) ],  n = N g,  n_eq = (T, u T, a_T T, 0, ...).
// F~ is Guo's source w_q [3 (c_q - u) + 9 (c_q.u) c_q].F, whose moments are the
// directional derivative of the equilibrium moments along F (M F~ = dm_eq/du . F at
// rho = 1).  M^-1 = M^T diag(1/|row|^2) because the rows are orthogonal.
//
// Instead of 19x19 matrix products, the forward and backward transforms are written in
// closed form over sums and differences of opposite populations, sharing sub-terms (the
// expression simplification of "GPU Optimization for High-Quality Kinetic Fluid
// Simulation", Eq. 10 and Table 2, applied to this basis): about 250 flops per D3Q19
// cell instead of ~1400.
#pragma once
#include "lbm_lattice.cuh"

namespace lbm {

struct CollideParams {
    float omega;    // BGK: 1/tau
    float fcoef;    // BGK: 1 - 1/(2 tau)
    float mA[19];   // MRT: s_k / |M_k|^2 (0 on conserved rows)
    float mB[19];   // MRT: (1 - s_k/2) / |M_k|^2 (1/|M_k|^2 on the momentum rows)
    float tA[7];    // thermal MRT: s_k / |N_k|^2
    float a_T;
    float gx, gy, gz;   // body acceleration
    float gbeta, T0;
    int up_axis;
    float cm[5];    // D3Q27 central moments: bulk rate, then the rates of orders 3, 4, 5, 6
};

// Body force and force-shifted velocity ([TLBM] Sec. 2).  ext: an additional force on the
// cell (the immersed boundary's), or null.
template <bool THERMAL>
LBM_HD void force_velocity(const CollideParams &P, float rho, float T, float jx, float jy,
                           float jz, float &Fx, float &Fy, float &Fz, float &ux, float &uy,
                           float &uz, const float *ext = nullptr)
{
    Fx = rho * P.gx;
    Fy = rho * P.gy;
    Fz = rho * P.gz;
    if (ext) {
        Fx += ext[0];
        Fy += ext[1];
        Fz += ext[2];
    }
    if (THERMAL) {
        const float b = rho * P.gbeta * (T - P.T0);
        if (P.up_axis == 0) Fx += b;
        else if (P.up_axis == 1) Fy += b;
        else Fz += b;
    }
    const float ir = 1.0f / rho;
    ux = (jx + 0.5f * Fx) * ir;
    uy = (jy + 0.5f * Fy) * ir;
    uz = (jz + 0.5f * Fz) * ir;
}

// ---------------------------------------------------------------- thermal MRT ---------

// D3Q7 rows: T; jx, jy, jz; e = -6 g0 + sum_k g_k; (0,2,2,-1,-1,-1,-1); (0,0,0,1,1,-1,-1).
// Norms 7, 2, 2, 2, 42, 12, 4.  Adds N^-1 d (d = per-row moment increments / norms).
LBM_HD void d3q7_add(float (&g)[7], float d0, float d1, float d2, float d3, float d4, float d5,
                     float d6)
{
    g[0] += d0 - 6.0f * d4;
    g[1] += d0 + d1 + d4 + 2.0f * d5;
    g[2] += d0 - d1 + d4 + 2.0f * d5;
    g[3] += d0 + d2 + d4 - d5 + d6;
    g[4] += d0 - d2 + d4 - d5 + d6;
    g[5] += d0 + d3 + d4 - d5 - d6;
    g[6] += d0 - d3 + d4 - d5 - d6;
}

LBM_HD void collide_d3q7(float (&g)[7], const CollideParams &P, float T, float ux, float uy,
                         float uz)
{
    const float s12 = g[1] + g[2], s34 = g[3] + g[4], s56 = g[5] + g[6];
    const float n1 = g[1] - g[2], n2 = g[3] - g[4], n3 = g[5] - g[6];
    const float n4 = -6.0f * g[0] + s12 + s34 + s56;
    const float n5 = 2.0f * s12 - s34 - s56;
    const float n6 = s34 - s56;
    d3q7_add(g, 0.0f, -P.tA[1] * (n1 - ux * T), -P.tA[2] * (n2 - uy * T),
             -P.tA[3] * (n3 - uz * T), -P.tA[4] * (n4 - P.a_T * T), -P.tA[5] * n5,
             -P.tA[6] * n6);
}

// D2Q5 (0, +x, +y, -x, -y) rows: T; jx; jy; e = -4 g0 + sum_k g_k; (0,1,-1,1,-1).
// Norms 5, 2, 2, 20, 4.
LBM_HD void d2q5_add(float (&g)[5], float d0, float d1, float d2, float d3, float d4)
{
    g[0] += d0 - 4.0f * d3;
    g[1] += d0 + d1 + d3 + d4;
    g[2] += d0 + d2 + d3 - d4;
    g[3] += d0 - d1 + d3 + d4;
    g[4] += d0 - d2 + d3 - d4;
}

LBM_HD void collide_d2q5(float (&g)[5], const CollideParams &P, float T, float ux, float uy)
{
    const float n1 = g[1] - g[3], n2 = g[2] - g[4];
    const float n3 = -4.0f * g[0] + g[1] + g[2] + g[3] + g[4];
    const float n4 = g[1] - g[2] + g[3] - g[4];
    d2q5_add(g, 0.0f, -P.tA[1] * (n1 - ux * T), -P.tA[2] * (n2 - uy * T),
             -P.tA[3] * (n3 - P.a_T * T), -P.tA[4] * n4);
}

// g_eq = N^-1 n_eq, n_eq = (T, u T, a_T T, 0, ...).
LBM_HD void d3q7_equilibrium(float (&g)[7], float a_T, float T, float ux, float uy, float uz)
{
    for (int k = 0; k < 7; ++k) g[k] = 0.0f;
    d3q7_add(g, T * (1.0f / 7.0f), 0.5f * ux * T, 0.5f * uy * T, 0.5f * uz * T,
             a_T * T * (1.0f / 42.0f), 0.0f, 0.0f);
}

LBM_HD void d2q5_equilibrium(float (&g)[5], float a_T, float T, float ux, float uy)
{
    for (int k = 0; k < 5; ++k) g[k] = 0.0f;
    d2q5_add(g, T * 0.2f, 0.5f * ux * T, 0.5f * uy * T, a_T * T * 0.05f, 0.0f);
}

// ------------------------------------------------------------------ D3Q19 MRT ---------

// d'Humieres basis rows: 0 rho, 1 e = 19c^2-30, 2 eps = (21c^4-53c^2+24)/2, 3/5/7 j,
// 4/6/8 q = (5c^2-9)c, 9 3pxx = 3cx^2-c^2, 10 3pixx = (3c^2-5)(3cx^2-c^2), 11 pww =
// cy^2-cz^2, 12 piww = (3c^2-5)(cy^2-cz^2), 13 pxy, 14 pyz, 15 pxz, 16-18 m.
// Norms 19, 2394, 252, 10, 40, 10, 40, 10, 40, 36, 72, 12, 24, 4, 4, 4, 8, 8, 8.
template <bool THERMAL, class TL>
LBM_HD void collide_d3q19_mrt(float (&f)[19], float (&g)[TL::QA], const CollideParams &P,
                              const float *ext)
{
    // sums and differences of opposite pairs
    const float sx = f[1] + f[2], dx = f[1] - f[2];
    const float sy = f[3] + f[4], dy = f[3] - f[4];
    const float sz = f[5] + f[6], dz = f[5] - f[6];
    const float a = f[7] + f[10], b = f[8] + f[9];            // xy edges (+,+)/(-,+) pairs
    const float exy1 = f[7] - f[10], exy2 = f[9] - f[8];      // along (1,1,0), (1,-1,0)
    const float c = f[11] + f[14], d = f[12] + f[13];          // xz edges
    const float exz1 = f[11] - f[14], exz2 = f[13] - f[12];   // along (1,0,1), (1,0,-1)
    const float e = f[15] + f[18], h = f[16] + f[17];          // yz edges
    const float eyz1 = f[15] - f[18], eyz2 = f[17] - f[16];   // along (0,1,1), (0,1,-1)
    const float X1 = exy1 + exy2, Y1 = exy1 - exy2;
    const float X2 = exz1 + exz2, Z2 = exz1 - exz2;
    const float Y3 = eyz1 + eyz2, Z3 = eyz1 - eyz2;
    const float Exy = a + b, Exz = c + d, Eyz = e + h;
    const float A = sx + sy + sz, E = Exy + Exz + Eyz;

    const float drho = f[0] + A + E;
    const float jx = dx + X1 + X2, jy = dy + Y1 + Y3, jz = dz + Z2 + Z3;
    float T = 0.0f;
    if constexpr (THERMAL) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) T += g[k];
    }
    const float rho = 1.0f + drho;
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<THERMAL>(P, rho, T, jx, jy, jz, Fx, Fy, Fz, ux, uy, uz, ext);

    // non-conserved moments of fbar
    const float m1 = -30.0f * f[0] - 11.0f * A + 8.0f * E;
    const float m2 = 12.0f * f[0] - 4.0f * A + E;
    const float m4 = -4.0f * dx + X1 + X2;
    const float m6 = -4.0f * dy + Y1 + Y3;
    const float m8 = -4.0f * dz + Z2 + Z3;
    const float ed = Exy + Exz - 2.0f * Eyz;
    const float m9 = 2.0f * sx - sy - sz + ed;
    const float m10 = -4.0f * sx + 2.0f * sy + 2.0f * sz + ed;
    const float ew = Exy - Exz;
    const float m11 = sy - sz + ew;
    const float m12 = -2.0f * sy + 2.0f * sz + ew;
    const float m13 = a - b, m14 = e - h, m15 = c - d;
    const float m16 = X1 - X2, m17 = Y3 - Y1, m18 = Z2 - Z3;

    // equilibrium moments (rest part removed from e and eps) and Guo source moments
    const float uxx = ux * ux, uyy = uy * uy, uzz = uz * uz;
    const float ru2 = rho * (uxx + uyy + uzz);
    const float uF = ux * Fx + uy * Fy + uz * Fz;
    const float p9 = rho * (2.0f * uxx - uyy - uzz), F9 = 2.0f * (2.0f * ux * Fx - uy * Fy - uz * Fz);
    const float p11 = rho * (uyy - uzz), F11 = 2.0f * (uy * Fy - uz * Fz);
    const float tt = 2.0f / 3.0f;

    const float D1 = P.mB[1] * (38.0f * uF) - P.mA[1] * (m1 - (-11.0f * drho + 19.0f * ru2));
    const float D2 = P.mB[2] * (-11.0f * uF) - P.mA[2] * (m2 - (3.0f * drho - 5.5f * ru2));
    const float D3 = P.mB[3] * Fx, D5 = P.mB[5] * Fy, D7 = P.mB[7] * Fz;
    const float D4 = P.mB[4] * (-tt * Fx) - P.mA[4] * (m4 + tt * rho * ux);
    const float D6 = P.mB[6] * (-tt * Fy) - P.mA[6] * (m6 + tt * rho * uy);
    const float D8 = P.mB[8] * (-tt * Fz) - P.mA[8] * (m8 + tt * rho * uz);
    const float D9 = P.mB[9] * F9 - P.mA[9] * (m9 - p9);
    const float D10 = P.mB[10] * (-0.5f * F9) - P.mA[10] * (m10 + 0.5f * p9);
    const float D11 = P.mB[11] * F11 - P.mA[11] * (m11 - p11);
    const float D12 = P.mB[12] * (-0.5f * F11) - P.mA[12] * (m12 + 0.5f * p11);
    const float D13 = P.mB[13] * (ux * Fy + uy * Fx) - P.mA[13] * (m13 - rho * ux * uy);
    const float D14 = P.mB[14] * (uy * Fz + uz * Fy) - P.mA[14] * (m14 - rho * uy * uz);
    const float D15 = P.mB[15] * (ux * Fz + uz * Fx) - P.mA[15] * (m15 - rho * ux * uz);
    const float D16 = -P.mA[16] * m16, D17 = -P.mA[17] * m17, D18 = -P.mA[18] * m18;

    // back transform, f += M^T D
    f[0] += -30.0f * D1 + 12.0f * D2;
    const float ba = -11.0f * D1 - 4.0f * D2;
    const float tx = D3 - 4.0f * D4, ty = D5 - 4.0f * D6, tz = D7 - 4.0f * D8;
    const float pxa = ba + 2.0f * D9 - 4.0f * D10;
    const float pya = ba - D9 + 2.0f * D10 + D11 - 2.0f * D12;
    const float pza = ba - D9 + 2.0f * D10 - D11 + 2.0f * D12;
    f[1] += pxa + tx;
    f[2] += pxa - tx;
    f[3] += pya + ty;
    f[4] += pya - ty;
    f[5] += pza + tz;
    f[6] += pza - tz;
    const float be = 8.0f * D1 + D2;
    const float exy = be + D9 + D10 + D11 + D12;
    const float exz = be + D9 + D10 - D11 - D12;
    const float eyz = be - 2.0f * D9 - 2.0f * D10;
    const float jxy = D3 + D4 + D16, jyx = D5 + D6 - D17;
    f[7] += exy + jxy + jyx + D13;
    f[10] += exy - jxy - jyx + D13;
    f[8] += exy - jxy + jyx - D13;
    f[9] += exy + jxy - jyx - D13;
    const float jxz = D3 + D4 - D16, jzx = D7 + D8 + D18;
    f[11] += exz + jxz + jzx + D15;
    f[14] += exz - jxz - jzx + D15;
    f[12] += exz - jxz + jzx - D15;
    f[13] += exz + jxz - jzx - D15;
    const float jyz = D5 + D6 + D17, jzy = D7 + D8 - D18;
    f[15] += eyz + jyz + jzy + D14;
    f[18] += eyz - jyz - jzy + D14;
    f[16] += eyz - jyz + jzy - D14;
    f[17] += eyz + jyz - jzy - D14;

    if constexpr (THERMAL) collide_d3q7(g, P, T, ux, uy, uz);
}

// ------------------------------------------------------------------- D2Q9 MRT ---------

// Lallemand-Luo basis: 0 rho, 1 e = 3c^2-4, 2 eps = (9c^4-21c^2+8)/2, 3 jx, 4 qx =
// (3c^2-5)cx, 5 jy, 6 qy, 7 pxx = cx^2-cy^2, 8 pxy.  Norms 9, 36, 36, 6, 12, 6, 12, 4, 4.
template <bool THERMAL, class TL>
LBM_HD void collide_d2q9_mrt(float (&f)[9], float (&g)[TL::QA], const CollideParams &P,
                             const float *ext)
{
    const float sx = f[1] + f[3], dx = f[1] - f[3];
    const float sy = f[2] + f[4], dy = f[2] - f[4];
    const float a = f[5] + f[7], b = f[6] + f[8];
    const float e1 = f[5] - f[7], e2 = f[8] - f[6];   // along (1,1), (1,-1)
    const float A = sx + sy, Dg = a + b;
    const float drho = f[0] + A + Dg;
    const float jx = dx + e1 + e2, jy = dy + e1 - e2;
    float T = 0.0f;
    if constexpr (THERMAL) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) T += g[k];
    }
    const float rho = 1.0f + drho;
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<THERMAL>(P, rho, T, jx, jy, 0.0f, Fx, Fy, Fz, ux, uy, uz, ext);

    const float m1 = -4.0f * f[0] - A + 2.0f * Dg;
    const float m2 = 4.0f * f[0] - 2.0f * A + Dg;
    const float m4 = -2.0f * dx + e1 + e2;
    const float m6 = -2.0f * dy + e1 - e2;
    const float m7 = sx - sy, m8 = a - b;
    const float uxx = ux * ux, uyy = uy * uy;
    const float ru2 = rho * (uxx + uyy);
    const float uF = ux * Fx + uy * Fy;

    const float D1 = P.mB[1] * (6.0f * uF) - P.mA[1] * (m1 - (-2.0f * drho + 3.0f * ru2));
    const float D2 = P.mB[2] * (-6.0f * uF) - P.mA[2] * (m2 - (drho - 3.0f * ru2));
    const float D3 = P.mB[3] * Fx, D5 = P.mB[5] * Fy;
    const float D4 = P.mB[4] * (-Fx) - P.mA[4] * (m4 + rho * ux);
    const float D6 = P.mB[6] * (-Fy) - P.mA[6] * (m6 + rho * uy);
    const float D7 = P.mB[7] * (2.0f * (ux * Fx - uy * Fy)) - P.mA[7] * (m7 - rho * (uxx - uyy));
    const float D8 = P.mB[8] * (ux * Fy + uy * Fx) - P.mA[8] * (m8 - rho * ux * uy);

    f[0] += -4.0f * D1 + 4.0f * D2;
    const float ba = -D1 - 2.0f * D2;
    const float tx = D3 - 2.0f * D4, ty = D5 - 2.0f * D6;
    f[1] += ba + tx + D7;
    f[3] += ba - tx + D7;
    f[2] += ba + ty - D7;
    f[4] += ba - ty - D7;
    const float bd = 2.0f * D1 + D2;
    const float jxd = D3 + D4, jyd = D5 + D6;
    f[5] += bd + jxd + jyd + D8;
    f[7] += bd - jxd - jyd + D8;
    f[6] += bd - jxd + jyd - D8;
    f[8] += bd + jxd - jyd - D8;

    if constexpr (THERMAL) collide_d2q5(g, P, T, ux, uy);
}

// ------------------------------------------------------------------------ BGK ---------

template <class L, bool THERMAL, class TL>
LBM_HD void collide_bgk(float (&f)[L::Q], float (&g)[TL::QA], const CollideParams &P,
                        const float *ext)
{
    float drho = 0.0f, jx = 0.0f, jy = 0.0f, jz = 0.0f;
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        drho += f[q];
        if (L::cx(q)) jx += L::cx(q) * f[q];
        if (L::cy(q)) jy += L::cy(q) * f[q];
        if (L::cz(q)) jz += L::cz(q) * f[q];
    }
    float T = 0.0f;
    if constexpr (THERMAL) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) T += g[k];
    }
    const float rho = 1.0f + drho;
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<THERMAL>(P, rho, T, jx, jy, jz, Fx, Fy, Fz, ux, uy, uz, ext);
    const float u15 = 1.5f * (ux * ux + uy * uy + uz * uz);
    const float uF3 = 3.0f * (ux * Fx + uy * Fy + uz * Fz);
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        const float cu = L::cx(q) * ux + L::cy(q) * uy + L::cz(q) * uz;
        const float cF = L::cx(q) * Fx + L::cy(q) * Fy + L::cz(q) * Fz;
        const float feq = L::w(q) * (drho + rho * (3.0f * cu + 4.5f * cu * cu - u15));
        const float src = L::w(q) * (3.0f * cF - uF3 + 9.0f * cu * cF);
        f[q] = f[q] - P.omega * (f[q] - feq) + P.fcoef * src;
    }
    if constexpr (THERMAL) {
        if constexpr (L::DIM == 3) collide_d3q7(g, P, T, ux, uy, uz);
        else collide_d2q5(g, P, T, ux, uy);
    }
}

// ------------------------------------------------- D3Q27 central-moment MRT ---------
//
// "GPU Optimization for High-Quality Kinetic Fluid Simulation", Sec. 3.1: D3Q27 (Fig. 2) and
// Omega = -M^-1 D (m - m_eq) (Eq. 5) with central moments, at fixed rates:
//   k_e = sum_q prod_a (c_qa - u_a)^e_a f_q,  e in {0,1,2}^3,  u = (j + F/2)/rho;
//   k_eq = rho prod_a mu[e_a], mu = (1, 0, 1/3) (a Maxwellian's central moments);
//   the source's central moments R_e = F_a prod_{b != a} mu[e_b] where e_a = 1;
//   k+ = k - s (k - k_eq) + (1 - s/2) R, with s = 0 on orders 0 and 1, the shear rate on
//   xy, xz, yz, xx - yy, xx - zz, the bulk rate on xx + yy + zz, one rate per order 3..6.
// The lattice is the tensor product of three D1Q3 stencils, so M(u) factors into 3-point
// transforms per axis, applied to the 3x3x3 array of populations: first the raw moments
// (f-, f0, f+) -> (sum f, sum c f, sum c^2 f) along x, y and z (u-independent: rho and j
// come out of it), then the shift of each axis to central moments about u_a (about 160
// flops in all instead of a 27 x 27 product).  The transform runs on the shifted
// populations fbar = f - w; the rest part's central moments, prod_a h[e_a] with
// h = (1, -u_a, 1/3 + u_a^2), enter the deviation k - k_eq analytically, so every quantity
// carried in fp32 is deviation-sized.

// (f-, f0, f+) -> raw moments (m0, m1, m2) = (sum f, sum c f, sum c^2 f), in place.
LBM_HD void cm_raw3(float &a, float &b, float &c)
{
    const float s = c + a, d = c - a;
    a = b + s;
    b = d;
    c = s;
}

// Raw moments (m0, m1, m2) -> central moments about u: k1 = m1 - u m0,
// k2 = m2 - 2 u m1 + u^2 m0 = m2 - u (m1 + k1), in place.
LBM_HD void cm_shift3(float &a, float &b, float &c, float u)
{
    const float k1 = fmaf(-u, a, b);
    c = fmaf(-u, b + k1, c);
    b = k1;
}

// (k0, k1, k2) about u -> (f-, f0, f+), in place: raw moments m1 = k1 + u k0,
// m2 = k2 + u (k1 + m1), then f0 = k0 - m2, f+- = (m2 +- m1) / 2.
LBM_HD void cm_backward3(float &a, float &b, float &c, float u)
{
    const float k0 = a, k1 = b, k2 = c;
    const float m1 = fmaf(u, k0, k1);
    const float m2 = fmaf(u, k1 + m1, k2);
    a = 0.5f * (m2 - m1);
    b = k0 - m2;
    c = 0.5f * (m2 + m1);
}

LBM_HD void collide_d3q27_cm(float (&f)[27], const CollideParams &P, const float *ext)
{
    using L = D3Q27;
    // a[z][y][x]: slot c + 1 of each axis, then (after the transforms) the exponent e
    float a[3][3][3];
#pragma unroll
    for (int q = 0; q < 27; ++q) a[L::cz(q) + 1][L::cy(q) + 1][L::cx(q) + 1] = f[q];
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_raw3(a[i][j][0], a[i][j][1], a[i][j][2]);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_raw3(a[i][0][j], a[i][1][j], a[i][2][j]);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_raw3(a[0][i][j], a[1][i][j], a[2][i][j]);
    // raw moments of fbar: sum fbar = rho - 1, sum c fbar = j
    const float rho = 1.0f + a[0][0][0];
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<false>(P, rho, 0.0f, a[0][0][1], a[0][1][0], a[1][0][0], Fx, Fy, Fz, ux, uy,
                          uz, ext);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_shift3(a[i][j][0], a[i][j][1], a[i][j][2], ux);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_shift3(a[i][0][j], a[i][1][j], a[i][2][j], uy);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_shift3(a[0][i][j], a[1][i][j], a[2][i][j], uz);
    // relaxation; h: central moments of the rest weights, mu: of the equilibrium per unit rho
    const float third = 1.0f / 3.0f;
    const float h[3][3] = {{1.0f, -ux, fmaf(ux, ux, third)},
                           {1.0f, -uy, fmaf(uy, uy, third)},
                           {1.0f, -uz, fmaf(uz, uz, third)}};
    constexpr float mu[3] = {1.0f, 0.0f, 1.0f / 3.0f};
    const float om = P.omega;
    // second-order normal moments: xx - yy, xx - zz at the shear rate, the trace at bulk
    {
        const float dxx = a[0][0][2] + (h[0][2] - rho * third);
        const float dyy = a[0][2][0] + (h[1][2] - rho * third);
        const float dzz = a[2][0][0] + (h[2][2] - rho * third);
        const float tr = P.cm[0] * (dxx + dyy + dzz);
        const float p = dxx - dyy, r = dxx - dzz;
        a[0][0][2] -= third * (tr + om * (p + r));
        a[0][2][0] -= third * (tr + om * (r - 2.0f * p));
        a[2][0][0] -= third * (tr + om * (p - 2.0f * r));
    }
#pragma unroll
    for (int ez = 0; ez < 3; ++ez)
#pragma unroll
        for (int ey = 0; ey < 3; ++ey)
#pragma unroll
            for (int ex = 0; ex < 3; ++ex) {
                const int n = ex + ey + ez;
                const int ones = (ex == 1) + (ey == 1) + (ez == 1);
                if (n == 0) continue;                       // rho
                if (n == 2 && ones == 0) continue;          // normal moments: done above
                float R = 0.0f;
                if (ex == 1) R += Fx * mu[ey] * mu[ez];
                if (ey == 1) R += Fy * mu[ex] * mu[ez];
                if (ez == 1) R += Fz * mu[ex] * mu[ey];
                float &k = a[ez][ey][ex];
                if (n == 1) {                               // momentum: conserved
                    k += R;
                    continue;
                }
                const float s = n == 2 ? om : P.cm[n - 2];
                const float dev = k + (h[0][ex] * h[1][ey] * h[2][ez] -
                                       rho * (mu[ex] * mu[ey] * mu[ez]));
                k = fmaf(-s, dev, k);
                if (ones == 1) k = fmaf(1.0f - 0.5f * s, R, k);
            }
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_backward3(a[0][i][j], a[1][i][j], a[2][i][j], uz);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_backward3(a[i][0][j], a[i][1][j], a[i][2][j], uy);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) cm_backward3(a[i][j][0], a[i][j][1], a[i][j][2], ux);
#pragma unroll
    for (int q = 0; q < 27; ++q) f[q] = a[L::cz(q) + 1][L::cy(q) + 1][L::cx(q) + 1];
}

// D3Q27 equilibrium rho prod_a phi(c_a, u_a), phi(0, u) = 2/3 - u^2, phi(+-1, u) =
// (1/3 + u^2 +- u)/2, returned shifted by w = prod_a phi(c_a, 0) as
// (prod phi - prod phi0) + drho prod phi, the first part telescoped so that no O(1) terms
// cancel in fp32.
LBM_HD float d3q27_feq_shifted(int cx, int cy, int cz, float drho, float ux, float uy, float uz)
{
    auto phi0 = [](int c) { return c == 0 ? 2.0f / 3.0f : 1.0f / 6.0f; };
    auto dphi = [](int c, float u) { return c == 0 ? -u * u : 0.5f * (u * u + c * u); };
    const float x0 = phi0(cx), y0 = phi0(cy), z0 = phi0(cz);
    const float dx = dphi(cx, ux), dy = dphi(cy, uy), dz = dphi(cz, uz);
    const float x = x0 + dx, y = y0 + dy;
    const float prod = x * y * (z0 + dz);
    const float tele = dx * y0 * z0 + x * dy * z0 + x * y * dz;
    return fmaf(drho, prod, tele);
}

// Dispatch on the collision model.  ext: additional force on the cell, or null.
template <class L, class TL, int COLL>
LBM_HD void collide(float (&f)[L::Q], float (&g)[TL::QA], const CollideParams &P,
                    const float *ext = nullptr)
{
    constexpr bool TH = TL::Q > 0;
    if constexpr (L::Q == 27) {
        (void)g;
        collide_d3q27_cm(f, P, ext);
    } else if (COLL == 0) {
        collide_bgk<L, TH, TL>(f, g, P, ext);
    } else if constexpr (L::Q == 19) {
        collide_d3q19_mrt<TH, TL>(f, g, P, ext);
    } else {
        collide_d2q9_mrt<TH, TL>(f, g, P, ext);
    }
}

}  // namespace lbm
