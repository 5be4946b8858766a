// Host emulation of the CUDA path's steps, for tests only (built by tests/conftest.py).
//
// Runs the library's own per-cell functions (cell_mask, init_cell, aa_step_cell,
// pull_step_cell, collide_in_place_cell, stream_cell, ib_sample, halo_cell) on the CPU, one cell at a
// time, but writes every step into a second buffer filled with NaN beforehand.  If a cell
// read a slot that another cell writes in the same step, or two cells wrote one slot, or a
// slot of a fluid cell were left unwritten, the stale or NaN value would reach the
// results; tests compare them with the oracle.
// The read-out uses the parity-aware logical load, as lbm_get_populations does.
#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <limits>
#include <memory>
#include <vector>

#include "lbm_setup.h"

using namespace lbm;

namespace {

// Run the masked AA steps without an immersed boundary with the mask loaded for every cell
// (the per-cell function's plain masked form) instead of computed outside the solid cells'
// box, as the kernels do; for tests that compare the two (emu_set_loaded_mask).
bool g_loaded_mask = false;

// Every population buffer carries GUARD NaN floats before and after its Q * S slots.  A read
// outside the slots yields NaN, which reaches the results; a write outside them is found by
// guards_intact() after every step.
constexpr size_t GUARD = 1024;

bool guards_intact(const std::vector<float> &v)
{
    for (size_t i = 0; i < GUARD; ++i)
        if (!std::isnan(v[i]) || !std::isnan(v[v.size() - 1 - i])) return false;
    return true;
}

// F: the mask computed from the coordinates outside the solid cells' box (boxed_mask), as
// the kernels do without an immersed boundary.
// I: the immersed-boundary form (cells with IB_BIT take the per-cell force).
template <class L, class TL, int C, bool M, bool O, bool NARROW, bool F, bool I>
void step_all(const Params &Pr, const Params &Pw)
{
    for (int z = 0; z < Pr.nz; ++z)
        for (int y = 0; y < Pr.ny; ++y)
            for (int x = 0; x < Pr.nx; ++x)
                aa_step_cell<L, TL, C, M, O, NARROW, I, F>(Pr, Pw, x, y, z);
}

// Two-buffer PULL step: pull from P.f, collide, natural store into W.
template <class L, class TL, int C, bool M, bool NARROW>
void pull_all(const Params &P, float *Wf, float *Wg)
{
    for (int z = 0; z < P.nz; ++z)
        for (int y = 0; y < P.ny; ++y)
            for (int x = 0; x < P.nx; ++x) pull_step_cell<L, TL, C, M, NARROW, M>(P, Wf, Wg, x, y, z);
}

// SPLIT step: collide in place, then pull from P.f into W.
template <class L, class TL, int C, bool M, bool NARROW>
void split_all(const Params &P, float *Wf, float *Wg)
{
    for (int i = 0; i < P.nx * P.ny * P.nz; ++i) collide_in_place_cell<L, TL, C, M, NARROW, M>(P, i);
    for (int z = 0; z < P.nz; ++z)
        for (int y = 0; y < P.ny; ++y)
            for (int x = 0; x < P.nx; ++x) stream_cell<L, TL, M, NARROW>(P, Wf, Wg, x, y, z);
}

template <class L, class TL, bool M, int O>
void read_all(const Params &P, float *fout, float *gout)
{
    const size_t N = (size_t)P.nx * P.ny * P.nz;
    for (int z = 0; z < P.nz; ++z)
        for (int y = 0; y < P.ny; ++y)
            for (int x = 0; x < P.nx; ++x) {
                const int idx = x + P.nx * (y + P.ny * z);
                uint32_t m = M ? P.mask[idx] : 0u;
                float f[L::Q], g[TL::QA];
                if (m & SKIP_BITS) {
                    for (int q = 0; q < L::Q; ++q) fout[q * N + idx] = 0.0f;
                    for (int k = 0; k < TL::Q; ++k) gout[k * N + idx] = 0.0f;
                    continue;
                }
                Offs o{};
                if (O != NATURAL) o = make_offs(x, y, z, P);
                load_cell<L, TL, M, O>(P, idx, o, m, f, g);
                for (int q = 0; q < L::Q; ++q) fout[q * N + idx] = f[q] + L::w(q);
                for (int k = 0; k < TL::Q; ++k) gout[k * N + idx] = g[k];
            }
}

// Immersed-boundary pass of one step on the host: the library's per-sample function, then
// a sequential scatter (the kernel uses atomic additions).
template <class L, class TL, int PAT>
void ib_all(const Params &P)
{
    for (int s = 0; s < P.ib_n; ++s) {
        int node[8];
        float K[8], gs[3];
        const int nn = ib_sample<L, TL, PAT>(P, s, node, K, gs);
        for (int a = 0; a < 3; ++a) P.ibg[a * P.ib_cap + s] = gs[a];
        for (int c = 0; c < nn; ++c) {
            if (P.mask[node[c]] & SOLID_BIT) continue;
            for (int a = 0; a < L::DIM; ++a) P.fib[(size_t)a * P.S + node[c]] += K[c] * gs[a];
        }
    }
}

template <class L, class TL>
void ib_pass(const Params &P, int pat)
{
    if (P.ib_n <= 0) return;
    if (pat == PULL) ib_all<L, TL, PULL>(P);
    else if (pat == AA_ODD) ib_all<L, TL, AA_ODD>(P);
    else ib_all<L, TL, NATURAL>(P);
}

// One domain's state on the host: population buffers (the current one and a NaN-filled one
// that each step writes), the link mask and the parameter block.
template <class L, class TL, int C, bool NARROW>
struct Domain {
    lbm_config cfg;
    lbm_setup::Layout Lay;
    std::vector<float> f, fn, g, gn;
    std::vector<uint32_t> mask;
    std::vector<char> ws;
    Params P{};
    int parity = 0;

    Domain(const lbm_config &c, const lbm_setup::Layout &lay) : cfg(c), Lay(lay)
    {
        const float nan = std::numeric_limits<float>::quiet_NaN();
        const size_t S = Lay.S;
        f.assign(Lay.Q * S + 2 * GUARD, nan);
        fn.assign(Lay.Q * S + 2 * GUARD, nan);
        g.assign((Lay.QT ? Lay.QT : 1) * S + 2 * GUARD, nan);
        gn.assign((Lay.QT ? Lay.QT : 1) * S + 2 * GUARD, nan);
        mask.assign(S, 0u);
        ws.resize(Lay.bytes + 256);
        lbm_setup::fill_params(cfg, Lay, ws.data(), P);
        point();
        P.mask = Lay.masked ? mask.data() : nullptr;
        if (Lay.masked)
            for (int z = 0; z < cfg.nz; ++z)
                for (int y = 0; y < cfg.ny; ++y)
                    for (int x = 0; x < cfg.nx; ++x) {
                        const uint32_t m = cell_mask<L, TL>(P, cfg.solid_mask, x, y, z);
                        const int idx = x + cfg.nx * (y + cfg.ny * z);
                        mask[idx] = m;
                        // the mask the kernels compute must equal the built one off the ghosts
                        if (Lay.ib_cap == 0 && !ghost_plane<L>(P, x, y, z) &&
                            boxed_mask<L, TL>(P, idx, x, y, z) != m)
                            ++face_mask_mismatches;
                    }
    }

    long long face_mask_mismatches = 0;

    void point()
    {
        P.f = f.data() + GUARD;
        P.g = Lay.QT ? g.data() + GUARD : nullptr;
    }

    long long guard_violations = 0;

    // immersed-boundary samples (given inside the domain) and their stencils' IB_BIT
    void set_ib(int ib_n, const float *ib_x, const float *ib_ub, const float *ib_w)
    {
        float *planes = const_cast<float *>(P.ibx);
        const size_t cap = P.ib_cap;
        for (int s = 0; s < ib_n; ++s) {
            for (int a = 0; a < 3; ++a) {
                planes[a * cap + s] = ib_x[3 * s + a];
                planes[(3 + a) * cap + s] = ib_ub ? ib_ub[3 * s + a] : 0.0f;
            }
            planes[6 * cap + s] = ib_w ? ib_w[s] : 1.0f;
            planes[7 * cap + s] = 1.0f;   // kept
        }
        P.ib_n = ib_n;
        const int n[3] = {cfg.nx, cfg.ny, cfg.nz};
        // the box of the stencil cells, as the marking kernel keeps it: {-lo, hi}
        int *box = const_cast<int *>(P.ib_box);
        for (int k = 0; k < 6; ++k) box[k] = std::numeric_limits<int>::min();
        for (int s = 0; s < ib_n; ++s) {
            int base[3] = {0, 0, 0};
            for (int a = 0; a < L::DIM; ++a) base[a] = (int)floorf(P.ibx[a * cap + s]);
            for (int c = 0; c < (1 << L::DIM); ++c) {
                int q[3] = {base[0], base[1], base[2]};
                for (int a = 0; a < L::DIM; ++a) {
                    q[a] += (c >> a) & 1;
                    if (q[a] >= n[a]) q[a] -= n[a];
                }
                mask[q[0] + cfg.nx * (q[1] + cfg.ny * q[2])] |= IB_BIT;
                for (int a = 0; a < 3; ++a) {
                    box[a] = std::max(box[a], -q[a]);
                    box[3 + a] = std::max(box[3 + a], q[a]);
                }
            }
        }
        // the mask the kernels compute must equal the built one at every cell
        for (int z = 0; z < cfg.nz; ++z)
            for (int y = 0; y < cfg.ny; ++y)
                for (int x = 0; x < cfg.nx; ++x) {
                    const int idx = x + cfg.nx * (y + cfg.ny * z);
                    if (boxed_mask<L, TL, true>(P, idx, x, y, z) != mask[idx])
                        ++face_mask_mismatches;
                }
    }

    void init(const float *rho, const float *u, const float *T)
    {
        for (int z = 0; z < cfg.nz; ++z)
            for (int y = 0; y < cfg.ny; ++y)
                for (int x = 0; x < cfg.nx; ++x) {
                    const int i = x + cfg.nx * (y + cfg.ny * z);
                    if (cfg.streaming == LBM_STREAM_PULL)
                        init_cell<L, TL, PULL>(P, i, rho, u, T, x, y, z);
                    else init_cell<L, TL, NATURAL>(P, i, rho, u, T, x, y, z);
                }
    }

    void step()
    {
        const int mode = cfg.streaming;
        const float nan = std::numeric_limits<float>::quiet_NaN();
        std::fill(fn.begin(), fn.end(), nan);
        std::fill(gn.begin(), gn.end(), nan);
        Params Pw = P;
        Pw.f = fn.data() + GUARD;
        Pw.g = Lay.QT ? gn.data() + GUARD : nullptr;
        float *wf = fn.data() + GUARD;
        float *wg = Lay.QT ? gn.data() + GUARD : nullptr;
        ib_pass<L, TL>(P, mode == LBM_STREAM_PULL    ? PULL
                          : mode == LBM_STREAM_SPLIT ? NATURAL
                          : parity                   ? AA_ODD
                                                     : NATURAL);
        if (mode == LBM_STREAM_PULL) {
            if (Lay.masked) pull_all<L, TL, C, true, NARROW>(P, wf, wg);
            else pull_all<L, TL, C, false, NARROW>(P, wf, wg);
        } else if (mode == LBM_STREAM_SPLIT) {
            if (Lay.masked) split_all<L, TL, C, true, NARROW>(P, wf, wg);
            else split_all<L, TL, C, false, NARROW>(P, wf, wg);
        } else if (Lay.masked && !g_loaded_mask) {
            // the kernels' form: the mask from the coordinates outside the box of the solid
            // cells and of the samples' stencil cells
            if (Lay.ib_cap > 0) {
                if (parity) step_all<L, TL, C, true, true, NARROW, true, true>(P, Pw);
                else step_all<L, TL, C, true, false, NARROW, true, true>(P, Pw);
            } else {
                if (parity) step_all<L, TL, C, true, true, NARROW, true, false>(P, Pw);
                else step_all<L, TL, C, true, false, NARROW, true, false>(P, Pw);
            }
        } else if (Lay.masked) {
            if (parity) step_all<L, TL, C, true, true, NARROW, false, true>(P, Pw);
            else step_all<L, TL, C, true, false, NARROW, false, true>(P, Pw);
        } else {
            if (parity) step_all<L, TL, C, false, true, NARROW, false, false>(P, Pw);
            else step_all<L, TL, C, false, false, NARROW, false, false>(P, Pw);
        }
        for (const auto *v : {&f, &fn, &g, &gn})
            if (!guards_intact(*v)) ++guard_violations;
        f.swap(fn);
        g.swap(gn);
        point();
        parity ^= 1;
    }

    // Logical populations (with the weights added back) of every cell.
    void read(float *fout, float *gout) const
    {
        const int pat = cfg.streaming == LBM_STREAM_PULL ? PULL
                        : (cfg.streaming == LBM_STREAM_AA && parity) ? AA_ODD : NATURAL;
        if (Lay.masked) {
            if (pat == PULL) read_all<L, TL, true, PULL>(P, fout, gout);
            else if (pat == AA_ODD) read_all<L, TL, true, AA_ODD>(P, fout, gout);
            else read_all<L, TL, true, NATURAL>(P, fout, gout);
        } else {
            if (pat == PULL) read_all<L, TL, false, PULL>(P, fout, gout);
            else if (pat == AA_ODD) read_all<L, TL, false, AA_ODD>(P, fout, gout);
            else read_all<L, TL, false, NATURAL>(P, fout, gout);
        }
    }

    // The library's per-cell halo function over one side's plane of an axis.
    void halo(int axis, int side, int phase, int unpack, float *buf)
    {
        const int n[3] = {cfg.nx, cfg.ny, cfg.nz};
        const int plane_cells = n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
        for (int i = 0; i < plane_cells; ++i)
            halo_cell<L, TL>(P, axis, side, phase, unpack, buf, i);
    }
};

template <class L, class TL, int C, bool NARROW>
int run(const lbm_config &cfg, const lbm_setup::Layout &Lay, const float *rho, const float *u,
        const float *T, int steps, float *fout, float *gout, uint32_t *mask_out, int ib_n,
        const float *ib_x, const float *ib_ub, const float *ib_w)
{
    Domain<L, TL, C, NARROW> d(cfg, Lay);
    if (d.face_mask_mismatches) return -30;
    if (Lay.ib_cap > 0) d.set_ib(ib_n, ib_x, ib_ub, ib_w);
    if (d.face_mask_mismatches) return -32;
    d.init(rho, u, T);
    for (int s = 0; s < steps; ++s) d.step();
    if (d.guard_violations) return -31;
    d.read(fout, gout);
    if (mask_out) std::memcpy(mask_out, d.mask.data(), sizeof(uint32_t) * (size_t)Lay.N);
    return 0;
}

// The domain split into slabs along its outer axis at planes edges[0..nslabs] (edges[0] =
// 0, edges[nslabs] = outer extent), each slab with a ghost plane per inner (or periodic)
// face, run with one halo exchange after every step (FILL after an even step, DRAIN after
// an odd one); the owned planes' logical populations are gathered into fout, gout.
template <class L, class TL, int C, bool NARROW>
int run_slabs(const lbm_config &cfg, const float *rho, const float *u, const float *T,
              int steps, int nslabs, const int *edges, float *fout, float *gout)
{
    using Dom = Domain<L, TL, C, NARROW>;
    const int dim = L::DIM, outer = dim - 1;
    const int n_outer = dim == 3 ? cfg.nz : cfg.ny;
    const int halo_dirs = L::Q == 27 ? 9 : (L::Q == 19 ? 5 : 3) + (TL::Q ? 1 : 0);
    const size_t plane = dim == 3 ? (size_t)cfg.nx * cfg.ny : (size_t)cfg.nx;
    const size_t N = (size_t)cfg.nx * cfg.ny * cfg.nz;
    const bool periodic = cfg.face_flow[2 * outer] == LBM_FACE_PERIODIC;
    std::vector<std::unique_ptr<Dom>> doms;
    std::vector<std::vector<int>> plane_lists;
    std::vector<std::vector<uint8_t>> solids;
    std::vector<std::array<bool, 2>> sides;
    std::vector<std::array<std::vector<float>, 2>> bufs;
    for (int r = 0; r < nslabs; ++r) {
        const int lo = edges[r], hi = edges[r + 1];
        const bool low = periodic || r > 0, high = periodic || r < nslabs - 1;
        std::vector<int> planes;
        if (low) planes.push_back((lo - 1 + n_outer) % n_outer);
        for (int p = lo; p < hi; ++p) planes.push_back(p);
        if (high) planes.push_back(hi % n_outer);
        lbm_config lc = cfg;
        if (dim == 3) lc.nz = (int)planes.size();
        else lc.ny = (int)planes.size();
        if (low) lc.face_flow[2 * outer] = LBM_FACE_HALO;
        if (high) lc.face_flow[2 * outer + 1] = LBM_FACE_HALO;
        const size_t Nl = plane * planes.size();
        std::vector<uint8_t> sol;
        std::vector<float> lr(Nl), lu((size_t)dim * Nl), lT(Nl);
        if (cfg.solid_mask) sol.resize(Nl);
        for (size_t k = 0; k < planes.size(); ++k)
            for (size_t i = 0; i < plane; ++i) {
                const size_t gi = (size_t)planes[k] * plane + i, li = k * plane + i;
                if (cfg.solid_mask) sol[li] = cfg.solid_mask[gi];
                lr[li] = rho[gi];
                for (int a = 0; a < dim; ++a) lu[a * Nl + li] = u[a * N + gi];
                if (T) lT[li] = T[gi];
            }
        lc.solid_mask = cfg.solid_mask ? sol.data() : nullptr;
        lbm_setup::Layout Lay;
        std::string why;
        if (lbm_setup::validate(&lc, &Lay, &why) != LBM_OK) return -10 - r;
        auto d = std::make_unique<Dom>(lc, Lay);
        if (d->face_mask_mismatches) return -40 - r;
        d->init(lr.data(), lu.data(), T ? lT.data() : nullptr);
        std::array<std::vector<float>, 2> b{std::vector<float>(halo_dirs * plane),
                                            std::vector<float>(halo_dirs * plane)};
        bufs.push_back(std::move(b));
        doms.push_back(std::move(d));
        plane_lists.push_back(planes);
        solids.push_back(std::move(sol));
        sides.push_back({low, high});
    }
    std::vector<std::pair<int, int>> pairs;
    for (int r = 0; r + 1 < nslabs; ++r) pairs.push_back({r, r + 1});
    if (periodic) pairs.push_back({nslabs - 1, 0});
    for (int s = 0; s < steps; ++s) {
        for (auto &d : doms) d->step();
        const int phase = doms[0]->parity == 1 ? LBM_HALO_FILL : LBM_HALO_DRAIN;
        for (auto [a, b] : pairs) {
            doms[a]->halo(outer, 1, phase, 0, bufs[a][1].data());
            doms[b]->halo(outer, 0, phase, 0, bufs[b][0].data());
        }
        for (auto [a, b] : pairs) {
            doms[a]->halo(outer, 1, phase, 1, bufs[b][0].data());
            doms[b]->halo(outer, 0, phase, 1, bufs[a][1].data());
        }
    }
    for (auto &d : doms)
        if (d->guard_violations) return -32;
    const int QT = TL::Q;
    for (int r = 0; r < nslabs; ++r) {
        const Dom &d = *doms[r];
        const size_t Nl = d.Lay.N;
        std::vector<float> lf((size_t)L::Q * Nl), lg((size_t)(QT ? QT : 1) * Nl);
        d.read(lf.data(), lg.data());
        const int first = sides[r][0] ? 1 : 0;
        for (int p = edges[r]; p < edges[r + 1]; ++p) {
            const size_t k = (size_t)(p - edges[r] + first);
            for (size_t i = 0; i < plane; ++i) {
                const size_t gi = (size_t)p * plane + i, li = k * plane + i;
                for (int q = 0; q < L::Q; ++q) fout[q * N + gi] = lf[q * Nl + li];
                for (int q = 0; q < QT; ++q) gout[q * N + gi] = lg[q * Nl + li];
            }
        }
    }
    return 0;
}

// The domain split into blocks: nb[a] pieces along axis a at planes edges[a][0..nb[a]].
// A block has a ghost plane at each face along a split axis that meets another block
// (every face of a split periodic axis).  After every step the blocks exchange axis by
// axis, z, then y, then x, each axis's unpacks done before the next axis's packs: a plane
// of a later axis includes the ghost rows that the earlier axes just filled or drained, so
// the populations of diagonal links reach the block across an edge or a corner in two or
// three hops.  The owned cells' logical populations are gathered into fout, gout.
template <class L, class TL, int C, bool NARROW>
int run_blocks(const lbm_config &cfg, const float *rho, const float *u, const float *T,
               int steps, const int *nb, const int *const *edges, int ordered, int swap,
               float *fout, float *gout)
{
    using Dom = Domain<L, TL, C, NARROW>;
    const int dim = L::DIM;
    const int n[3] = {cfg.nx, cfg.ny, cfg.nz};
    const size_t N = (size_t)n[0] * n[1] * n[2];
    const int halo_dirs = L::Q == 27 ? 9 : (L::Q == 19 ? 5 : 3) + (TL::Q ? 1 : 0);
    const int nblocks = nb[0] * nb[1] * nb[2];
    struct Block {
        std::unique_ptr<Dom> d;
        std::vector<int> coords[3];   // global coordinate of each local index, per axis
        int bi[3], owned_lo[3], owned_hi[3], ext[3];
        bool low[3], high[3];
        std::vector<uint8_t> sol;
    };
    std::vector<Block> blocks(nblocks);
    auto block_at = [&](int i, int j, int k) { return i + nb[0] * (j + nb[1] * k); };
    for (int b = 0; b < nblocks; ++b) {
        Block &B = blocks[b];
        B.bi[0] = b % nb[0];
        B.bi[1] = (b / nb[0]) % nb[1];
        B.bi[2] = b / (nb[0] * nb[1]);
        lbm_config lc = cfg;
        for (int a = 0; a < 3; ++a) {
            const bool split = a < dim && nb[a] > 1;
            const bool periodic = cfg.face_flow[2 * a] == LBM_FACE_PERIODIC;
            const int lo = split ? edges[a][B.bi[a]] : 0;
            const int hi = split ? edges[a][B.bi[a] + 1] : n[a];
            B.low[a] = split && (periodic || B.bi[a] > 0);
            B.high[a] = split && (periodic || B.bi[a] < nb[a] - 1);
            if (B.low[a]) B.coords[a].push_back((lo - 1 + n[a]) % n[a]);
            for (int p = lo; p < hi; ++p) B.coords[a].push_back(p);
            if (B.high[a]) B.coords[a].push_back(hi % n[a]);
            B.ext[a] = (int)B.coords[a].size();
            B.owned_lo[a] = B.low[a] ? 1 : 0;
            B.owned_hi[a] = B.owned_lo[a] + (hi - lo);
            if (B.low[a]) lc.face_flow[2 * a] = LBM_FACE_HALO;
            if (B.high[a]) lc.face_flow[2 * a + 1] = LBM_FACE_HALO;
        }
        lc.nx = B.ext[0];
        lc.ny = B.ext[1];
        lc.nz = B.ext[2];
        const size_t Nl = (size_t)B.ext[0] * B.ext[1] * B.ext[2];
        std::vector<float> lr(Nl), lu((size_t)dim * Nl), lT(Nl);
        if (cfg.solid_mask) B.sol.resize(Nl);
        for (int k = 0; k < B.ext[2]; ++k)
            for (int j = 0; j < B.ext[1]; ++j)
                for (int i = 0; i < B.ext[0]; ++i) {
                    const size_t li = i + (size_t)B.ext[0] * (j + (size_t)B.ext[1] * k);
                    const size_t gi = B.coords[0][i] +
                                      (size_t)n[0] * (B.coords[1][j] + (size_t)n[1] * B.coords[2][k]);
                    if (cfg.solid_mask) B.sol[li] = cfg.solid_mask[gi];
                    lr[li] = rho[gi];
                    for (int a = 0; a < dim; ++a) lu[a * Nl + li] = u[a * N + gi];
                    if (T) lT[li] = T[gi];
                }
        lc.solid_mask = cfg.solid_mask ? B.sol.data() : nullptr;
        lbm_setup::Layout Lay;
        std::string why;
        if (lbm_setup::validate(&lc, &Lay, &why) != LBM_OK) return -10 - b;
        B.d = std::make_unique<Dom>(lc, Lay);
        if (B.d->face_mask_mismatches) return -40 - b;
        B.d->init(lr.data(), lu.data(), T ? lT.data() : nullptr);
    }
    // one axis's packed buffers: (lower block, upper block, [lower's high side, upper's low])
    struct Exchange {
        int axis, lo, hi;
        std::array<std::vector<float>, 2> buf;
    };
    for (int s = 0; s < steps; ++s) {
        for (auto &B : blocks) B.d->step();
        const int phase = blocks[0].d->parity == 1 ? LBM_HALO_FILL : LBM_HALO_DRAIN;
        std::vector<Exchange> held;   // ordered == 0: every axis packs before any unpacks
        auto unpack = [&](std::vector<Exchange> &xs) {
            for (auto &x : xs) {
                blocks[x.lo].d->halo(x.axis, 1, phase, 1, x.buf[1].data());
                blocks[x.hi].d->halo(x.axis, 0, phase, 1, x.buf[0].data());
            }
        };
        for (int a = dim - 1; a >= 0; --a) {
            if (nb[a] < 2) continue;
            if (swap) {   // the buffer-free form, one face after another
                for (int b = 0; b < nblocks; ++b) {
                    const Block &B = blocks[b];
                    if (!B.high[a]) continue;
                    int j[3] = {B.bi[0], B.bi[1], B.bi[2]};
                    j[a] = (j[a] + 1) % nb[a];
                    const Block &H = blocks[block_at(j[0], j[1], j[2])];
                    const int u0 = a == 0 ? 1 : 0, v0 = a == 2 ? 1 : 2;
                    const int cells = B.ext[u0] * B.ext[v0];
                    for (int i = 0; i < cells; ++i)
                        halo_swap_cell<L, TL>(B.d->P, H.d->P, a, phase, i);
                }
                continue;
            }
            // pairs (block, its high neighbour along a), with the wrap on a periodic axis
            std::vector<std::pair<int, int>> pairs;
            for (int b = 0; b < nblocks; ++b) {
                const Block &B = blocks[b];
                if (!B.high[a]) continue;
                int j[3] = {B.bi[0], B.bi[1], B.bi[2]};
                j[a] = (j[a] + 1) % nb[a];
                pairs.push_back({b, block_at(j[0], j[1], j[2])});
            }
            const int u0 = a == 0 ? 1 : 0, v0 = a == 2 ? 1 : 2;
            std::vector<Exchange> xs;
            for (const auto [lo, hi] : pairs) {
                const Block &B = blocks[lo];
                const size_t cells = (size_t)B.ext[u0] * B.ext[v0];
                Exchange x{a, lo, hi, {}};
                x.buf[0].assign(halo_dirs * cells, 0.0f);
                x.buf[1].assign(halo_dirs * cells, 0.0f);
                blocks[lo].d->halo(a, 1, phase, 0, x.buf[0].data());
                blocks[hi].d->halo(a, 0, phase, 0, x.buf[1].data());
                xs.push_back(std::move(x));
            }
            if (ordered) unpack(xs);
            else for (auto &x : xs) held.push_back(std::move(x));
        }
        unpack(held);
    }
    const int QT = TL::Q;
    for (const Block &B : blocks) {
        if (B.d->guard_violations) return -32;
        const size_t Nl = B.d->Lay.N;
        std::vector<float> lf((size_t)L::Q * Nl), lg((size_t)(QT ? QT : 1) * Nl);
        B.d->read(lf.data(), lg.data());
        for (int k = B.owned_lo[2]; k < B.owned_hi[2]; ++k)
            for (int j = B.owned_lo[1]; j < B.owned_hi[1]; ++j)
                for (int i = B.owned_lo[0]; i < B.owned_hi[0]; ++i) {
                    const size_t li = i + (size_t)B.ext[0] * (j + (size_t)B.ext[1] * k);
                    const size_t gi = B.coords[0][i] +
                                      (size_t)n[0] * (B.coords[1][j] + (size_t)n[1] * B.coords[2][k]);
                    for (int q = 0; q < L::Q; ++q) fout[q * N + gi] = lf[q * Nl + li];
                    for (int q = 0; q < QT; ++q) gout[q * N + gi] = lg[q * Nl + li];
                }
    }
    return 0;
}

// Read and write sets of one AA step, brute force on a tiny grid.  W(c): the slots cell c
// writes, found by stepping c alone into a NaN-filled buffer.  R(c): the slots whose value
// reaches c's outputs, found by poisoning each slot of the state with NaN in turn.  The step
// is race-free in place when R(c) == W(c) for every cell and no slot lies in two cells' W.
// The step runs in the form the kernels use (F: mask from the coordinates outside the solid
// cells' box).  Returns the number of violations.
template <class L, class TL, int C, bool M, bool F, bool O>
long long race_violations(Domain<L, TL, C, true> &d)
{
    const float nan = std::numeric_limits<float>::quiet_NaN();
    const Params Pr = d.P;
    Params Pw = d.P;
    std::vector<float> wf(d.f.size()), wg(d.g.size());
    Pw.f = wf.data() + GUARD;
    Pw.g = d.Lay.QT ? wg.data() + GUARD : nullptr;
    std::vector<int> owner_f(wf.size(), -1), owner_g(wg.size(), -1);
    long long bad = 0;
    std::vector<size_t> Wf, Wg;
    auto step_cell = [&](int x, int y, int z) {
        std::fill(wf.begin(), wf.end(), nan);
        std::fill(wg.begin(), wg.end(), nan);
        aa_step_cell<L, TL, C, M, O, true, M && !F, F>(Pr, Pw, x, y, z);
    };
    auto outputs_poisoned = [&]() {
        for (size_t s : Wf)
            if (std::isnan(wf[s])) return true;
        for (size_t s : Wg)
            if (std::isnan(wg[s])) return true;
        return false;
    };
    auto read_set_check = [&](std::vector<float> &state, const std::vector<size_t> &W, int x,
                              int y, int z) {
        for (size_t s = 0; s < state.size(); ++s) {
            const float keep = state[s];
            state[s] = nan;
            step_cell(x, y, z);
            const bool read = outputs_poisoned();
            state[s] = keep;
            const bool written = std::binary_search(W.begin(), W.end(), s);
            if (read != written) ++bad;
        }
    };
    for (int z = 0; z < d.cfg.nz; ++z)
        for (int y = 0; y < d.cfg.ny; ++y)
            for (int x = 0; x < d.cfg.nx; ++x) {
                const int c = x + d.cfg.nx * (y + d.cfg.ny * z);
                step_cell(x, y, z);
                Wf.clear();
                Wg.clear();
                for (size_t s = 0; s < wf.size(); ++s)
                    if (!std::isnan(wf[s])) Wf.push_back(s);
                if (d.Lay.QT)
                    for (size_t s = 0; s < wg.size(); ++s)
                        if (!std::isnan(wg[s])) Wg.push_back(s);
                for (size_t s : Wf) {
                    if (owner_f[s] >= 0) ++bad;
                    owner_f[s] = c;
                }
                for (size_t s : Wg) {
                    if (owner_g[s] >= 0) ++bad;
                    owner_g[s] = c;
                }
                read_set_check(d.f, Wf, x, y, z);
                if (d.Lay.QT) read_set_check(d.g, Wg, x, y, z);
            }
    return bad;
}

template <class L, class TL, int C>
long long race_any(const lbm_config &cfg, const lbm_setup::Layout &Lay, bool odd)
{
    Domain<L, TL, C, true> d(cfg, Lay);
    if (d.face_mask_mismatches) return -30;
    const size_t N = (size_t)Lay.N;
    std::vector<float> rho(N), u(3 * N), T(N);
    for (size_t i = 0; i < N; ++i) {
        rho[i] = 1.0f + 1e-3f * (float)(i % 7);
        for (int a = 0; a < 3; ++a) u[a * N + i] = 0.01f * (float)((i + 3 * a) % 5) - 0.02f;
        T[i] = 0.05f * (float)(i % 3);
    }
    d.init(rho.data(), u.data(), T.data());
    const bool M = Lay.masked, F = Lay.masked && Lay.ib_cap == 0;
    if (!M) return odd ? race_violations<L, TL, C, false, false, true>(d)
                       : race_violations<L, TL, C, false, false, false>(d);
    if (F) return odd ? race_violations<L, TL, C, true, true, true>(d)
                      : race_violations<L, TL, C, true, true, false>(d);
    return odd ? race_violations<L, TL, C, true, false, true>(d)
               : race_violations<L, TL, C, true, false, false>(d);
}

// Overlap of a slab's or block's halo exchange with the next step's interior (the drivers'
// overlapped order): the exchange after a step -- FILL before an odd step, DRAIN before an
// even one, over every HALO face of every axis -- runs beside the next step's launch over
// the box of cells [ilo, ihi).  Brute force on a tiny grid: the packs' read set (each slot holds its own index; the
// buffer shows which were read), the unpack's write set (a sentinel buffer), and, for every
// interior cell of the next step, its write set (stepped alone into a NaN-filled buffer) and
// which of the packs' and unpacks' slots it reads (each such slot poisoned in turn).  The
// overlap is race-free when no interior cell reads or writes a slot a pack reads or an
// unpack writes.  Returns the number of such (cell, slot) pairs.
template <class L, class TL, int C, bool M, bool F, bool O>
long long overlap_pairs(Domain<L, TL, C, true> &d, const int *ilo, const int *ihi)
{
    const float nan = std::numeric_limits<float>::quiet_NaN();
    const int phase = O ? LBM_HALO_FILL : LBM_HALO_DRAIN;
    const int n[3] = {d.cfg.nx, d.cfg.ny, d.cfg.nz};
    const int ndir = L::Q == 27 ? 9 : (L::Q == 19 ? 5 : 3) + (TL::Q ? 1 : 0);
    // slots: f slot s as s, g slot s as -1 - s (indices into the vectors, guards included)
    std::vector<long long> touched;
    const std::vector<float> f0 = d.f, g0 = d.g;
    for (int face = 0; face < 2 * L::DIM; ++face) {
        const int axis = face / 2, side = face % 2;
        if (d.cfg.face_flow[face] != LBM_FACE_HALO) continue;
        const int plane_cells = n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
        std::vector<float> buf((size_t)ndir * plane_cells);
        for (size_t i = 0; i < d.f.size(); ++i) d.f[i] = (float)i;
        for (size_t i = 0; i < d.g.size(); ++i) d.g[i] = -1.0f - (float)i;
        std::fill(buf.begin(), buf.end(), nan);
        d.halo(axis, side, phase, 0, buf.data());
        for (float v : buf)
            if (!std::isnan(v)) touched.push_back((long long)v);
        d.f = f0;
        d.g = g0;
        d.point();
        const float mark = 1.0e30f;
        std::fill(buf.begin(), buf.end(), mark);
        for (auto *v : {&d.f, &d.g}) std::fill(v->begin(), v->end(), 0.0f);
        d.halo(axis, side, phase, 1, buf.data());
        for (size_t i = 0; i < d.f.size(); ++i)
            if (d.f[i] == mark) touched.push_back((long long)i);
        for (size_t i = 0; i < d.g.size(); ++i)
            if (d.g[i] == mark) touched.push_back(-1 - (long long)i);
        d.f = f0;
        d.g = g0;
        d.point();
    }
    std::sort(touched.begin(), touched.end());
    touched.erase(std::unique(touched.begin(), touched.end()), touched.end());
    if (touched.empty()) return -50;   // nothing exchanged: the check would be vacuous
    std::vector<float> wf(d.f.size()), wg(d.g.size());
    Params Pw = d.P;
    Pw.f = wf.data() + GUARD;
    Pw.g = d.Lay.QT ? wg.data() + GUARD : nullptr;
    auto step_cell = [&](int x, int y, int z) {
        std::fill(wf.begin(), wf.end(), nan);
        std::fill(wg.begin(), wg.end(), nan);
        aa_step_cell<L, TL, C, M, O, true, M && !F, F>(d.P, Pw, x, y, z);
    };
    auto slot_ref = [&](std::vector<float> &fv, std::vector<float> &gv, long long t) -> float & {
        return t >= 0 ? fv[(size_t)t] : gv[(size_t)(-1 - t)];
    };
    long long bad = 0;
    for (int z = 0; z < d.cfg.nz; ++z)
        for (int y = 0; y < d.cfg.ny; ++y)
            for (int x = 0; x < d.cfg.nx; ++x) {
                const int c3[3] = {x, y, z};
                bool inside = true;
                for (int a = 0; a < 3; ++a) inside = inside && c3[a] >= ilo[a] && c3[a] < ihi[a];
                if (!inside) continue;
                step_cell(x, y, z);
                std::vector<size_t> Wf, Wg;
                for (size_t i = 0; i < wf.size(); ++i)
                    if (!std::isnan(wf[i])) Wf.push_back(i);
                for (size_t i = 0; i < wg.size(); ++i)
                    if (!std::isnan(wg[i]) && d.Lay.QT) Wg.push_back(i);
                for (long long t : touched) {
                    if (!std::isnan(slot_ref(wf, wg, t))) {   // written by the cell
                        ++bad;
                        continue;
                    }
                    float &st = slot_ref(d.f, d.g, t);
                    const float keep = st;
                    st = nan;
                    step_cell(x, y, z);
                    st = keep;
                    bool read = false;
                    for (size_t i : Wf) read = read || std::isnan(wf[i]);
                    for (size_t i : Wg) read = read || std::isnan(wg[i]);
                    if (read) ++bad;
                }
            }
    return bad;
}

template <class L, class TL, int C>
long long overlap_any(const lbm_config &cfg, const lbm_setup::Layout &Lay, bool next_odd,
                      const int *ilo, const int *ihi)
{
    Domain<L, TL, C, true> d(cfg, Lay);
    if (d.face_mask_mismatches) return -30;
    const size_t N = (size_t)Lay.N;
    std::vector<float> rho(N), u(3 * N), T(N);
    for (size_t i = 0; i < N; ++i) {
        rho[i] = 1.0f + 1e-3f * (float)(i % 7);
        for (int a = 0; a < 3; ++a) u[a * N + i] = 0.01f * (float)((i + 3 * a) % 5) - 0.02f;
        T[i] = 0.05f * (float)(i % 3);
    }
    d.init(rho.data(), u.data(), T.data());
    const bool M = Lay.masked, F = Lay.masked && Lay.ib_cap == 0;
    if (!M) return next_odd ? overlap_pairs<L, TL, C, false, false, true>(d, ilo, ihi)
                            : overlap_pairs<L, TL, C, false, false, false>(d, ilo, ihi);
    if (F) return next_odd ? overlap_pairs<L, TL, C, true, true, true>(d, ilo, ihi)
                           : overlap_pairs<L, TL, C, true, true, false>(d, ilo, ihi);
    return next_odd ? overlap_pairs<L, TL, C, true, false, true>(d, ilo, ihi)
                    : overlap_pairs<L, TL, C, true, false, false>(d, ilo, ihi);
}

}  // namespace

// Violations of race-freedom of one AA step (even: odd = 0) on a tiny grid, see
// race_violations; negative on a bad configuration.
extern "C" long long emu_race_violations(const lbm_config *cfg, int odd)
{
    lbm_setup::Layout Lay;
    std::string why;
    if (lbm_setup::validate(cfg, &Lay, &why) != LBM_OK) return -1;
    if (cfg->streaming != LBM_STREAM_AA) return -2;
    const bool mrt = cfg->collision == LBM_MRT, o = odd != 0;
    if (cfg->lattice == 27) return race_any<D3Q27, NoThermal, 2>(*cfg, Lay, o);
    if (cfg->lattice == 19) {
        if (cfg->thermal == 7)
            return mrt ? race_any<D3Q19, D3Q7, 1>(*cfg, Lay, o) : race_any<D3Q19, D3Q7, 0>(*cfg, Lay, o);
        return mrt ? race_any<D3Q19, NoThermal, 1>(*cfg, Lay, o)
                   : race_any<D3Q19, NoThermal, 0>(*cfg, Lay, o);
    }
    if (cfg->thermal == 5)
        return mrt ? race_any<D2Q9, D2Q5, 1>(*cfg, Lay, o) : race_any<D2Q9, D2Q5, 0>(*cfg, Lay, o);
    return mrt ? race_any<D2Q9, NoThermal, 1>(*cfg, Lay, o) : race_any<D2Q9, NoThermal, 0>(*cfg, Lay, o);
}

template <bool NARROW>
int run_any(const lbm_config *cfg, const lbm_setup::Layout &Lay, const float *rho,
            const float *u, const float *T, int steps, float *fout, float *gout,
            uint32_t *mask_out, int ib_n, const float *ib_x, const float *ib_ub,
            const float *ib_w)
{
    const bool mrt = cfg->collision == LBM_MRT;
    if (cfg->lattice == 27)
        return run<D3Q27, NoThermal, 2, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w);
    if (cfg->lattice == 19) {
        if (cfg->thermal == 7)
            return mrt ? run<D3Q19, D3Q7, 1, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w)
                       : run<D3Q19, D3Q7, 0, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w);
        return mrt ? run<D3Q19, NoThermal, 1, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w)
                   : run<D3Q19, NoThermal, 0, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w);
    }
    if (cfg->thermal == 5)
        return mrt ? run<D2Q9, D2Q5, 1, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w)
                   : run<D2Q9, D2Q5, 0, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w);
    return mrt ? run<D2Q9, NoThermal, 1, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w)
               : run<D2Q9, NoThermal, 0, NARROW>(*cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x, ib_ub, ib_w);
}

extern "C" void emu_set_loaded_mask(int on) { g_loaded_mask = on != 0; }

// narrow != 0: the step uses 32-bit population indices, as the library does whenever
// every index fits in 32 bits; 0: the 64-bit form used for larger grids.
extern "C" int emu_run(const lbm_config *cfg, const float *rho, const float *u, const float *T,
                       int steps, float *fout, float *gout, uint32_t *mask_out, int narrow,
                       int ib_n, const float *ib_x, const float *ib_ub, const float *ib_w)
{
    lbm_setup::Layout Lay;
    std::string why;
    if (lbm_setup::validate(cfg, &Lay, &why) != LBM_OK) return -1;
    if (ib_n > Lay.ib_cap) return -2;
    return narrow ? run_any<true>(cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n, ib_x,
                                  ib_ub, ib_w)
                  : run_any<false>(cfg, Lay, rho, u, T, steps, fout, gout, mask_out, ib_n,
                                   ib_x, ib_ub, ib_w);
}

// Slab decomposition of the whole domain cfg (AA layout), see run_slabs; the same
// population read-out as emu_run.
extern "C" int emu_run_slabs(const lbm_config *cfg, const float *rho, const float *u,
                             const float *T, int steps, int nslabs, const int *edges,
                             float *fout, float *gout)
{
    lbm_setup::Layout Lay;
    std::string why;
    if (lbm_setup::validate(cfg, &Lay, &why) != LBM_OK) return -1;
    if (cfg->streaming != LBM_STREAM_AA || nslabs < 1) return -2;
    const bool mrt = cfg->collision == LBM_MRT;
    if (cfg->lattice == 27)
        return run_slabs<D3Q27, NoThermal, 2, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout);
    if (cfg->lattice == 19) {
        if (cfg->thermal == 7)
            return mrt ? run_slabs<D3Q19, D3Q7, 1, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout)
                       : run_slabs<D3Q19, D3Q7, 0, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout);
        return mrt ? run_slabs<D3Q19, NoThermal, 1, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout)
                   : run_slabs<D3Q19, NoThermal, 0, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout);
    }
    if (cfg->thermal == 5)
        return mrt ? run_slabs<D2Q9, D2Q5, 1, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout)
                   : run_slabs<D2Q9, D2Q5, 0, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout);
    return mrt ? run_slabs<D2Q9, NoThermal, 1, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout)
               : run_slabs<D2Q9, NoThermal, 0, true>(*cfg, rho, u, T, steps, nslabs, edges, fout, gout);
}

// Block decomposition of the whole domain cfg (AA layout), see run_blocks: nb[3] pieces per
// axis, edges the concatenated plane lists (nb[0] + 1 entries for x, then y, then z).
// ordered = 0 packs every axis before any unpack (the diagonal hops then have nothing to
// carry): a negative control for the tests.  swap = 1 moves each face with halo_swap_cell
// (no buffer) instead of a pack and an unpack.
extern "C" int emu_run_blocks(const lbm_config *cfg, const float *rho, const float *u,
                              const float *T, int steps, const int *nb, const int *edges,
                              int ordered, int swap, float *fout, float *gout)
{
    lbm_setup::Layout Lay;
    std::string why;
    if (lbm_setup::validate(cfg, &Lay, &why) != LBM_OK) return -1;
    if (cfg->streaming != LBM_STREAM_AA) return -2;
    for (int a = 0; a < 3; ++a)
        if (nb[a] < 1) return -3;
    const int *e[3] = {edges, edges + nb[0] + 1, edges + nb[0] + nb[1] + 2};
    const bool mrt = cfg->collision == LBM_MRT;
#define LBM_EMU_BLOCKS(Lt, Tt, Ct) run_blocks<Lt, Tt, Ct, true>(*cfg, rho, u, T, steps, nb, e, ordered, swap, fout, gout)
    if (cfg->lattice == 27) return LBM_EMU_BLOCKS(D3Q27, NoThermal, 2);
    if (cfg->lattice == 19) {
        if (cfg->thermal == 7)
            return mrt ? LBM_EMU_BLOCKS(D3Q19, D3Q7, 1) : LBM_EMU_BLOCKS(D3Q19, D3Q7, 0);
        return mrt ? LBM_EMU_BLOCKS(D3Q19, NoThermal, 1) : LBM_EMU_BLOCKS(D3Q19, NoThermal, 0);
    }
    if (cfg->thermal == 5)
        return mrt ? LBM_EMU_BLOCKS(D2Q9, D2Q5, 1) : LBM_EMU_BLOCKS(D2Q9, D2Q5, 0);
    return mrt ? LBM_EMU_BLOCKS(D2Q9, NoThermal, 1) : LBM_EMU_BLOCKS(D2Q9, NoThermal, 0);
#undef LBM_EMU_BLOCKS
}

// div_by against the quotient for divisor d at the numerators n_lo .. n_hi (inclusive) and at
// every multiple of d, and one below it, up to 2^31 - 1 (at most `multiples` of them):
// returns the number of wrong quotients.
extern "C" long long emu_divisor_errors(unsigned d, unsigned n_lo, unsigned n_hi,
                                        long long multiples)
{
    const Divisor dv = lbm_setup::divisor(d);
    long long bad = 0;
    for (unsigned long long n = n_lo; n <= n_hi; ++n)
        bad += div_by((unsigned)n, dv) != (unsigned)(n / d);
    const unsigned long long top = (1ull << 31) - 1;
    const unsigned long long step = std::max<unsigned long long>(
        d, (top / d / (unsigned long long)std::max<long long>(multiples, 1)) * d);
    for (unsigned long long k = d; k <= top; k += step)
        for (unsigned long long n : {k - 1, k, std::min(k + d - 1, top)})
            bad += div_by((unsigned)n, dv) != (unsigned)(n / d);
    bad += div_by((unsigned)top, dv) != (unsigned)(top / d);
    return bad;
}

// The linear AA launch's cell mapping over the planes [lo, hi) of a grid (3-D: one grid row
// per plane, threads along the plane; 2-D: threads along the rows [lo, hi)): every thread
// index below the range's cell count names a distinct cell of those planes, in storage order,
// and the next index none.  Returns the number of violations.
extern "C" long long emu_linear_mapping_errors(int dim, int nx, int ny, int nz, int lo, int hi)
{
    // the whole grid takes the plain form (no box), a range of planes the box form
    const bool box = !(lo == 0 && hi == (dim == 3 ? nz : ny));
    Params P{};
    P.nx = nx;
    P.ny = ny;
    P.nz = nz;
    P.run_lo[0] = P.run_lo[1] = P.run_lo[2] = 0;
    P.run_hi[0] = nx;
    P.run_hi[1] = ny;
    P.run_hi[2] = nz;
    P.run_lo[dim - 1] = lo;
    P.run_hi[dim - 1] = hi;
    P.linear = 1;
    P.div_nx = lbm_setup::divisor((unsigned)nx);
    long long bad = 0;
    auto check = [&](bool in, int x, int y, int z, long long want) {
        const long long idx = x + (long long)nx * (y + (long long)ny * z);
        bad += !in || x < 0 || x >= nx || y < 0 || y >= ny || z < 0 || z >= nz || idx != want;
    };
    if (dim == 3) {
        const long long plane = (long long)nx * ny;
        for (int p = 0; p < hi - lo; ++p) {
            for (long long t = 0; t <= plane; ++t) {
                int x = -1, y = -1, z = -1;
                const bool in = (box ? linear_cell_coords<D3Q19, true>(P, (int)t, p, x, y, z)
                                       : linear_cell_coords<D3Q19, false>(P, (int)t, p, x, y, z));
                if (t == plane) bad += in;
                else check(in, x, y, z, (lo + p) * plane + t);
            }
        }
    } else {
        const long long cells = (long long)nx * (hi - lo);
        for (long long t = 0; t <= cells; ++t) {
            int x = -1, y = -1, z = -1;
            const bool in = (box ? linear_cell_coords<D2Q9, true>(P, (int)t, 0, x, y, z)
                                       : linear_cell_coords<D2Q9, false>(P, (int)t, 0, x, y, z));
            if (t == cells) bad += in;
            else check(in, x, y, z, (long long)lo * nx + t);
        }
    }
    return bad;
}

// Every neighbour index the odd-step access pattern forms (idx + offset of +-c_q for each
// direction, with the periodic wrap) must name a cell of the grid: returns the number of
// out-of-range indices over all cells (0 expected).
extern "C" long long emu_count_bad_indices(int lattice, int nx, int ny, int nz)
{
    Params P{};
    P.nx = nx;
    P.ny = ny;
    P.nz = nz;
    const long long N = (long long)nx * ny * nz;
    long long bad = 0;
    for (int z = 0; z < nz; ++z)
        for (int y = 0; y < ny; ++y)
            for (int x = 0; x < nx; ++x) {
                const long long idx = x + (long long)nx * (y + (long long)ny * z);
                const Offs o = make_offs(x, y, z, P);
                const int Q = lattice;
                for (int q = 0; q < Q; ++q) {
                    const int cx = lattice == 27 ? D3Q27::cx(q) : lattice == 19 ? D3Q19::cx(q) : D2Q9::cx(q);
                    const int cy = lattice == 27 ? D3Q27::cy(q) : lattice == 19 ? D3Q19::cy(q) : D2Q9::cy(q);
                    const int cz = lattice == 27 ? D3Q27::cz(q) : lattice == 19 ? D3Q19::cz(q) : D2Q9::cz(q);
                    for (int sgn = -1; sgn <= 1; sgn += 2) {
                        const long long j = idx + nb(o, sgn * cx, sgn * cy, sgn * cz);
                        if (j < 0 || j >= N) ++bad;
                    }
                }
            }
    return bad;
}

// (cell, slot) pairs by which the next step's launch over the box of cells [ilo, ihi) would
// race with the exchange before it, every HALO face of every axis (see overlap_pairs);
// next_odd: the next step is odd (the exchange is a FILL), else even (a DRAIN).  Negative on
// a bad configuration.
extern "C" long long emu_box_overlap_violations(const lbm_config *cfg, int next_odd,
                                                const int *ilo, const int *ihi)
{
    lbm_setup::Layout Lay;
    std::string why;
    if (lbm_setup::validate(cfg, &Lay, &why) != LBM_OK) return -1;
    if (cfg->streaming != LBM_STREAM_AA || !Lay.halo) return -2;
    const bool mrt = cfg->collision == LBM_MRT, o = next_odd != 0;
    if (cfg->lattice == 27) return overlap_any<D3Q27, NoThermal, 2>(*cfg, Lay, o, ilo, ihi);
    if (cfg->lattice == 19) {
        if (cfg->thermal == 7)
            return mrt ? overlap_any<D3Q19, D3Q7, 1>(*cfg, Lay, o, ilo, ihi)
                       : overlap_any<D3Q19, D3Q7, 0>(*cfg, Lay, o, ilo, ihi);
        return mrt ? overlap_any<D3Q19, NoThermal, 1>(*cfg, Lay, o, ilo, ihi)
                   : overlap_any<D3Q19, NoThermal, 0>(*cfg, Lay, o, ilo, ihi);
    }
    if (cfg->thermal == 5)
        return mrt ? overlap_any<D2Q9, D2Q5, 1>(*cfg, Lay, o, ilo, ihi)
                   : overlap_any<D2Q9, D2Q5, 0>(*cfg, Lay, o, ilo, ihi);
    return mrt ? overlap_any<D2Q9, NoThermal, 1>(*cfg, Lay, o, ilo, ihi)
               : overlap_any<D2Q9, NoThermal, 0>(*cfg, Lay, o, ilo, ihi);
}

// The same for a launch over the whole outer-axis planes [ilo, ihi) (the slab overlap).
extern "C" long long emu_overlap_violations(const lbm_config *cfg, int next_odd, int ilo,
                                            int ihi)
{
    const int dim = cfg->lattice == 9 ? 2 : 3;
    int lo[3] = {0, 0, 0}, hi[3] = {cfg->nx, cfg->ny, cfg->nz};
    lo[dim - 1] = ilo;
    hi[dim - 1] = ihi;
    return emu_box_overlap_violations(cfg, next_odd, lo, hi);
}
