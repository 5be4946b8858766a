// Host-side set-up shared by the C ABI: validation of an lbm_config, the workspace
// layout, and the kernel parameters (rates scaled by the moment-row norms, anti-bounce-
// back weights, face flags).
#pragma once
#include <cmath>
#include <cstdint>
#include <string>

#include "../../include/lbm.h"
#include "lbm_internal.h"

namespace lbm_setup {

constexpr size_t ALIGN = 256;
inline size_t align_up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }

// Norms |row|^2 of the moment bases (rows as listed in include/lbm.h).
constexpr double NORM_D3Q19[19] = {19, 2394, 252, 10, 40, 10, 40, 10, 40, 36,
                               72, 12,   24,  4,  4,  4,  8,  8,  8};
constexpr double NORM_D2Q9[9] = {9, 36, 36, 6, 12, 6, 12, 4, 4};
constexpr double NORM_D3Q7[7] = {7, 2, 2, 2, 42, 12, 4};
constexpr double NORM_D2Q5[5] = {5, 2, 2, 20, 4};

inline bool conserved_row(int lattice, int k)
{
    return k == 0 || k == 3 || k == 5 || (lattice == 19 && k == 7);
}

struct Layout {
    int Q = 0, QT = 0, dim = 0;
    long long N = 0;
    size_t S = 0;
    bool masked = false, has_solid = false;
    // Without an immersed boundary, the masked AA step kernels compute a cell's link mask
    // from its coordinates (its wall faces) and load it only inside box_lo..box_hi: the
    // bounding box of the solid cells widened by one cell, empty without solid cells.
    int box_lo[3] = {0, 0, 0}, box_hi[3] = {-1, -1, -1};
    int streaming = LBM_STREAM_AA;
    bool halo = false;
    size_t off_f = 0, off_g = 0, off_f2 = 0, off_g2 = 0, off_mask = 0, off_solid = 0;
    size_t off_partial = 0, off_result = 0, off_fib = 0, off_ib = 0, off_ibsort = 0;
    size_t off_ibbox = 0;
    int ib_cap = 0;
    size_t bytes = 0;
};

// Bounding box (inclusive) of the solid cells of c->solid_mask, widened by one cell on each
// side: every cell with a link into a solid cell, and every solid cell, lies inside it.  An
// axis on which the widened range leaves the grid through a periodic face is taken whole
// (the neighbour across the face is at the other end); otherwise the range is clipped to
// the grid.  Empty (lo > hi) when no cell is solid.
inline void solid_box(const lbm_config *c, int lo[3], int hi[3])
{
    const int n[3] = {c->nx, c->ny, c->nz};
    int l[3] = {n[0], n[1], n[2]}, h[3] = {-1, -1, -1};
    const uint8_t *s = c->solid_mask;
    size_t i = 0;
    for (int z = 0; z < n[2]; ++z)
        for (int y = 0; y < n[1]; ++y)
            for (int x = 0; x < n[0]; ++x, ++i) {
                if (!s[i]) continue;
                const int p[3] = {x, y, z};
                for (int a = 0; a < 3; ++a) {
                    l[a] = p[a] < l[a] ? p[a] : l[a];
                    h[a] = p[a] > h[a] ? p[a] : h[a];
                }
            }
    for (int a = 0; a < 3; ++a) {
        lo[a] = 0;
        hi[a] = -1;
    }
    if (h[0] < 0) return;
    for (int a = 0; a < 3; ++a) {
        int wl = l[a] - 1, wh = h[a] + 1;
        if ((wl < 0 || wh > n[a] - 1) && c->face_flow[2 * a] == LBM_FACE_PERIODIC) {
            wl = 0;
            wh = n[a] - 1;
        }
        lo[a] = wl < 0 ? 0 : wl;
        hi[a] = wh > n[a] - 1 ? n[a] - 1 : wh;
    }
}

inline lbm_status validate(const lbm_config *c, Layout *L, std::string *why)
{
    auto bad = [&](lbm_status s, const char *msg) {
        *why = msg;
        return s;
    };
    if (!c) return bad(LBM_ERR_ARG, "config is NULL");
    if (c->lattice != LBM_D3Q19 && c->lattice != LBM_D2Q9 && c->lattice != LBM_D3Q27)
        return bad(LBM_ERR_ARG, "lattice must be LBM_D3Q19, LBM_D2Q9 or LBM_D3Q27");
    if (c->thermal != LBM_THERMAL_NONE && c->thermal != LBM_D3Q7 && c->thermal != LBM_D2Q5)
        return bad(LBM_ERR_ARG, "thermal must be NONE, LBM_D3Q7 or LBM_D2Q5");
    if ((c->thermal == LBM_D3Q7 && c->lattice != LBM_D3Q19) ||
        (c->thermal == LBM_D2Q5 && c->lattice != LBM_D2Q9))
        return bad(LBM_ERR_UNSUPPORTED, "thermal lattice must match: D3Q19+D3Q7 or D2Q9+D2Q5");
    if (c->collision != LBM_BGK && c->collision != LBM_MRT && c->collision != LBM_CM)
        return bad(LBM_ERR_ARG, "collision must be LBM_BGK, LBM_MRT or LBM_CM");
    if ((c->lattice == LBM_D3Q27) != (c->collision == LBM_CM))
        return bad(LBM_ERR_UNSUPPORTED, "D3Q27 goes with LBM_CM, and LBM_CM with D3Q27 only");
    if (c->lattice == LBM_D3Q27) {
        if (!(std::isfinite(c->tau) && c->tau > 0.5))
            return bad(LBM_ERR_ARG, "tau must be finite and > 1/2");
        for (int k = 0; k < 5; ++k)
            if (!(c->cm_rates[k] > 0.0 && c->cm_rates[k] < 2.0))
                return bad(LBM_ERR_ARG, "central-moment rates must lie in (0, 2)");
        if (c->thermal != LBM_THERMAL_NONE)
            return bad(LBM_ERR_UNSUPPORTED, "D3Q27 takes no thermal lattice");
        if (c->streaming != LBM_STREAM_AA)
            return bad(LBM_ERR_UNSUPPORTED, "D3Q27 runs the AA layout only");
    }
    if (c->nx < 1 || c->ny < 1 || c->nz < 1) return bad(LBM_ERR_ARG, "grid sizes must be >= 1");
    if (c->lattice == LBM_D2Q9 && c->nz != 1) return bad(LBM_ERR_ARG, "D2Q9 needs nz == 1");
    const long long N = (long long)c->nx * c->ny * c->nz;
    if (N >= (1LL << 31)) return bad(LBM_ERR_ARG, "nx*ny*nz must be < 2^31");
    if (c->nz > 65535) return bad(LBM_ERR_UNSUPPORTED, "nz must be <= 65535");
    if (lbm::cell_shape(c->nx, c->ny, c->nz).grid.y > 65535)
        return bad(LBM_ERR_UNSUPPORTED,
                   "ny too large: ny / (rows per block) must be <= 65535 (ny <= 65535 once nx > 32)");
    if (c->collision == LBM_BGK && !(std::isfinite(c->tau) && c->tau > 0.5))
        return bad(LBM_ERR_ARG, "BGK tau must be finite and > 1/2");
    const int Q = c->lattice;
    if (c->collision == LBM_MRT)
        for (int k = 0; k < Q; ++k)
            if (!conserved_row(Q, k) && !(c->s[k] >= 0.0 && c->s[k] < 2.0))
                return bad(LBM_ERR_ARG, "MRT rates of non-conserved rows must lie in [0, 2)");
    const int QT = c->thermal;
    if (QT) {
        for (int k = 1; k < QT; ++k)
            if (!(c->s_T[k] >= 0.0 && c->s_T[k] < 2.0))
                return bad(LBM_ERR_ARG, "thermal rates must lie in [0, 2)");
        if (!(c->a_T > -(QT - 1) && c->a_T < 1.0))
            return bad(LBM_ERR_ARG, "a_T must lie in (-(Q_T - 1), 1)");
    } else if (c->gbeta != 0.0) {
        return bad(LBM_ERR_ARG, "buoyancy (gbeta != 0) needs a thermal lattice");
    }
    const int dim = (Q == LBM_D2Q9) ? 2 : 3;
    if (c->up_axis < 0 || c->up_axis >= dim) return bad(LBM_ERR_ARG, "up_axis out of range");
    if (dim == 2 && c->g_body[2] != 0.0) return bad(LBM_ERR_ARG, "g_body[2] must be 0 in 2-D");
    for (int a = 0; a < 3; ++a)
        if (!std::isfinite(c->g_body[a])) return bad(LBM_ERR_ARG, "g_body must be finite");
    if (!std::isfinite(c->gbeta) || !std::isfinite(c->T0))
        return bad(LBM_ERR_ARG, "gbeta and T0 must be finite");
    bool any_wall = false, any_halo = false;
    for (int i = 0; i < 2 * dim; ++i) {
        const int k = c->face_flow[i];
        if (k != LBM_FACE_PERIODIC && k != LBM_FACE_WALL && k != LBM_FACE_HALO)
            return bad(LBM_ERR_ARG, "face_flow entries must be PERIODIC, WALL or HALO");
        if (c->face_T[i] != LBM_TFACE_ADIABATIC && c->face_T[i] != LBM_TFACE_DIRICHLET)
            return bad(LBM_ERR_ARG, "face_T entries must be ADIABATIC or DIRICHLET");
        if (!std::isfinite(c->T_wall[i])) return bad(LBM_ERR_ARG, "T_wall must be finite");
        any_wall |= k == LBM_FACE_WALL;
        any_halo |= k == LBM_FACE_HALO;
    }
    for (int a = 0; a < dim; ++a) {
        const int lo = c->face_flow[2 * a], hi = c->face_flow[2 * a + 1];
        // a wrap must pair with a wrap; walls and halos mix (no slot is claimed twice)
        if ((lo == LBM_FACE_PERIODIC) != (hi == LBM_FACE_PERIODIC))
            return bad(LBM_ERR_UNSUPPORTED,
                       "both faces of an axis must have the same flow kind (AA addressing)");
    }
    if (any_halo) {
        const int n[3] = {c->nx, c->ny, c->nz};
        for (int a = 0; a < dim; ++a) {
            const int ghosts = (c->face_flow[2 * a] == LBM_FACE_HALO) +
                               (c->face_flow[2 * a + 1] == LBM_FACE_HALO);
            if (n[a] < ghosts + 1)
                return bad(LBM_ERR_ARG,
                           "a slab or block needs at least one owned plane besides its ghosts");
        }
        if (c->streaming != LBM_STREAM_AA)
            return bad(LBM_ERR_UNSUPPORTED, "HALO faces need the AA layout");
        if (c->ib_max_samples > 0)
            return bad(LBM_ERR_UNSUPPORTED, "HALO faces with immersed-boundary samples");
    }
    L->Q = Q;
    L->QT = QT;
    L->dim = dim;
    L->N = N;
    L->S = ((size_t)N + 63) / 64 * 64;
    L->has_solid = c->solid_mask != nullptr;
    L->ib_cap = c->ib_max_samples;
    // a slab's ghost planes are found by their coordinate: HALO faces need no mask
    L->masked = any_wall || L->has_solid || L->ib_cap > 0;
    if (L->has_solid) solid_box(c, L->box_lo, L->box_hi);
    L->halo = any_halo;
    size_t off = 0;
    L->off_f = off;
    off = align_up(off + (size_t)Q * L->S * sizeof(float));
    L->off_g = off;
    off = align_up(off + (size_t)QT * L->S * sizeof(float));
    L->streaming = c->streaming;
    L->off_f2 = L->off_g2 = off;
    if (c->streaming != LBM_STREAM_AA) {
        off = align_up(off + (size_t)Q * L->S * sizeof(float));
        L->off_g2 = off;
        off = align_up(off + (size_t)QT * L->S * sizeof(float));
    }
    L->off_mask = off;
    if (L->masked) off = align_up(off + L->S * sizeof(uint32_t));
    L->off_solid = off;
    if (L->has_solid) off = align_up(off + L->S);
    L->off_fib = L->off_ib = off;
    if (L->ib_cap > 0) {
        off = align_up(off + 3 * L->S * sizeof(float));   // per-cell force
        L->off_ib = off;
        off = align_up(off + (size_t)11 * L->ib_cap * sizeof(float));   // x3 ub3 w kept g3
        L->off_ibsort = off;   // device ordering of samples (lbm_set_ib_samples_device)
        off = align_up(off + lbm::ib_order_scratch_bytes(L->ib_cap));
        L->off_ibbox = off;    // box of the samples' stencil cells (6 ints)
        off = align_up(off + 6 * sizeof(int));
    }
    L->off_partial = off;
    off = align_up(off + (size_t)lbm::DIAG_BLOCKS * lbm::DIAG_N * sizeof(double));
    L->off_result = off;
    off = align_up(off + lbm::DIAG_N * sizeof(double));
    L->bytes = off;
    return LBM_OK;
}

// The multiplier and shift of lbm::div_by for divisor d >= 1.
inline lbm::Divisor divisor(unsigned d)
{
    int l = 0;
    while ((1ull << l) < d) ++l;
    lbm::Divisor r;
    r.s = 31 + l;
    r.m = ((1ull << r.s) + d - 1) / d;
    return r;
}

inline void fill_params(const lbm_config &g, const Layout &L, char *ws, lbm::Params &P)
{
    P.f = reinterpret_cast<float *>(ws + L.off_f);
    P.g = L.QT ? reinterpret_cast<float *>(ws + L.off_g) : nullptr;
    P.fib = L.ib_cap ? reinterpret_cast<float *>(ws + L.off_fib) : nullptr;
    float *ib = L.ib_cap ? reinterpret_cast<float *>(ws + L.off_ib) : nullptr;
    P.ib_cap = L.ib_cap;
    P.ib_n = 0;
    P.ibx = ib;
    P.ibub = ib ? ib + 3 * (size_t)L.ib_cap : nullptr;
    P.ibw = ib ? ib + 6 * (size_t)L.ib_cap : nullptr;
    P.ibg = ib ? ib + 8 * (size_t)L.ib_cap : nullptr;   // plane 7: 1 = kept, 0 = dropped
    P.ib_box = L.ib_cap ? reinterpret_cast<const int *>(ws + L.off_ibbox) : nullptr;
    const bool two = L.streaming != LBM_STREAM_AA;
    P.fo = two ? reinterpret_cast<float *>(ws + L.off_f2) : nullptr;
    P.go = (two && L.QT) ? reinterpret_cast<float *>(ws + L.off_g2) : nullptr;
    P.mask = L.masked ? reinterpret_cast<const uint32_t *>(ws + L.off_mask) : nullptr;
    P.S = L.S;
    P.nx = g.nx;
    P.ny = g.ny;
    P.nz = g.nz;
    lbm::CollideParams &C = P.c;
    C.omega = (float)(1.0 / g.tau);
    C.fcoef = (float)(1.0 - 0.5 / g.tau);
    const double *norm = (g.lattice == LBM_D3Q19) ? NORM_D3Q19 : NORM_D2Q9;
    for (int k = 0; k < 19; ++k) {
        C.mA[k] = 0.0f;
        C.mB[k] = 0.0f;
    }
    for (int k = 0; k < 5; ++k) C.cm[k] = g.lattice == LBM_D3Q27 ? (float)g.cm_rates[k] : 0.0f;
    for (int k = 0; k < (g.lattice == LBM_D3Q27 ? 0 : g.lattice); ++k) {
        if (k == 0) continue;
        if (conserved_row(g.lattice, k)) {
            C.mB[k] = (float)(1.0 / norm[k]);
        } else if (g.collision == LBM_MRT) {
            C.mA[k] = (float)(g.s[k] / norm[k]);
            C.mB[k] = (float)((1.0 - 0.5 * g.s[k]) / norm[k]);
        }
    }
    for (int k = 0; k < 7; ++k) C.tA[k] = 0.0f;
    const double *tnorm = (g.thermal == LBM_D3Q7) ? NORM_D3Q7 : NORM_D2Q5;
    for (int k = 1; k < g.thermal; ++k) C.tA[k] = (float)(g.s_T[k] / tnorm[k]);
    C.a_T = (float)g.a_T;
    C.gx = (float)g.g_body[0];
    C.gy = (float)g.g_body[1];
    C.gz = (float)g.g_body[2];
    C.gbeta = (float)g.gbeta;
    C.T0 = (float)g.T0;
    C.up_axis = g.up_axis;
    const int dim = L.dim;
    for (int i = 0; i < 6; ++i) {
        const bool active = i < 2 * dim;
        P.face_wall[i] = active && g.face_flow[i] == LBM_FACE_WALL;
        P.face_halo[i] = active && g.face_flow[i] == LBM_FACE_HALO;
        P.face_dir[i] = P.face_wall[i] && g.thermal && g.face_T[i] == LBM_TFACE_DIRICHLET;
        P.T_wall[i] = (float)g.T_wall[i];
    }
    const int outer = dim - 1, n_outer = dim == 3 ? g.nz : g.ny;
    for (int a = 0; a < 3; ++a) {
        P.box_lo[a] = L.box_lo[a];
        P.box_hi[a] = L.box_hi[a];
    }
    P.ghost_lo = P.face_halo[2 * outer] ? 0 : -1;
    P.ghost_hi = P.face_halo[2 * outer + 1] ? n_outer - 1 : -1;
    const int ext[3] = {g.nx, g.ny, g.nz};
    P.ghost_inner = 0;
    for (int a = 0; a < 3; ++a) {
        P.ghost3_lo[a] = P.face_halo[2 * a] ? 0 : -1;
        P.ghost3_hi[a] = P.face_halo[2 * a + 1] ? ext[a] - 1 : -1;
        if (a != outer && (P.face_halo[2 * a] || P.face_halo[2 * a + 1])) P.ghost_inner = 1;
    }
    for (int a = 0; a < 3; ++a) {
        P.run_lo[a] = 0;
        P.run_hi[a] = ext[a];
    }
    P.linear = g.nx % 32 != 0;
    P.div_nx = divisor((unsigned)g.nx);
    // anti-bounce-back weight omega = (4 + a_T)/10 (D2Q5) or (6 + a_T)/21 (D3Q7)
    const double omega = (g.thermal == LBM_D2Q5) ? (4.0 + g.a_T) / 10.0 : (6.0 + g.a_T) / 21.0;
    for (int k = 0; k < 7; ++k) P.abbT[k] = 0.0f;
    for (int k = 1; k < g.thermal; ++k) {
        const int cx = (g.lattice == 19) ? lbm::D3Q19::cx(k) : lbm::D2Q9::cx(k);
        const int cy = (g.lattice == 19) ? lbm::D3Q19::cy(k) : lbm::D2Q9::cy(k);
        const int cz = (g.lattice == 19) ? lbm::D3Q19::cz(k) : lbm::D2Q9::cz(k);
        P.abbT[k] = (float)(omega * g.T_wall[lbm::axis_face(cx, cy, cz)]);
    }
}

}  // namespace lbm_setup
