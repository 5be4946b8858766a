// Kernels of the CUDA path: the fused AA collide-and-stream step (even and odd forms)
// and the auxiliary kernels (equilibrium initialisation, link-mask build, parity-aware
// read-out of macroscopic fields and populations, diagnostics reduction).
//
// Storage ("Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI",
// Sec. 3, SoA index x + Nx y + Nx Ny z + Nx Ny Nz i): population q of cell idx lives at
// f[q * S + idx], S = plane stride (cells rounded up to 64, so that every plane starts
// on a 256-byte boundary); f holds f_q - w_q (see lbm_collide.cuh), g holds g_q.
//
// AA pattern ("GPU lattice Boltzmann: streaming layout and performance"): one buffer.
//   even step: read (q, x); collide; write f+_q to (opp q, x).
//   odd step:  read (opp q, x - c_q); collide; write f+_q to (q, x + c_q).
// Wall links fold into the odd step through the per-cell link mask (bit q: the link
// from x along c_q ends on a wall or a solid cell): the read of q redirects to the own
// slot (q, x) when link opp q is a wall, the write of q redirects to (opp q, x) when
// link q is a wall.  Both hit the same slot, so every cell writes exactly the slots it
// read and no cells race.  This realises the half-way bounce-back f_qbar(x, t+1) =
// f_q+(x, t) and, for Dirichlet thermal links, the anti-bounce-back g_qbar(x, t+1) =
// -g_q+(x, t) + omega T_w (multi-GPU thermal LBM page, Sec. 2): the sign flip and the
// omega T_w term are applied where the odd step writes, or reads, the redirected slot.
// Even steps need no wall handling.  After an odd number of steps the logical state is
// read with the odd step's read pattern.
//
// Two-buffer modes (that page's A-B layout, for comparison): PULL fuses the step into one
// kernel that pulls f_q(x - c_q) (bounce-back f_opp(x) on wall links) from the current
// buffer, collides and writes (q, x) of the other buffer, so the stored state is the
// post-collision one and is read with the pull pattern; SPLIT collides in place (natural
// slots), then a second kernel pulls into the other buffer, so the stored state is the
// natural pre-collision one (304 B per D3Q19 update instead of 152).
#pragma once
#include <climits>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "lbm_collide.cuh"

namespace lbm {

// Division of 0 <= n < 2^31 by an invariant d >= 1 with one multiply and one shift
// (Granlund and Montgomery, "Division by invariant integers using multiplication", 1994):
// m = ceil(2^s / d) with s = 31 + ceil(log2 d).  floor(n m / 2^s) = floor(n / d) because the
// excess n (m d - 2^s) / (d 2^s) stays below 1/d: m d - 2^s < d <= 2^(s-31) and n < 2^31.
// m <= 2^32, so n m fits in 64 bits.
struct Divisor {
    unsigned long long m;
    int s;
};

LBM_HD unsigned div_by(unsigned n, const Divisor &d)
{
    return (unsigned)(((unsigned long long)n * d.m) >> d.s);
}

struct Params {
    float *f;              // Q planes of S floats (shifted populations), current buffer
    float *g;              // Q_T planes (thermal), may be null
    float *fo, *go;        // the other buffer of the two-buffer modes (null for AA)
    const uint32_t *mask;  // link mask, null when there are no walls or solids
    size_t S;              // plane stride in elements
    int nx, ny, nz;
    CollideParams c;
    float abbT[7];         // per thermal direction k: omega * T_wall of the face k leaves by
    int face_wall[6];      // per face: 1 = wall (flow)
    int face_halo[6];      // per face: 1 = halo face of a slab (ghost plane, no wrap)
    int ghost_lo, ghost_hi;  // outer-axis coordinate of a slab's ghost planes, -1 = none
    // blocks: ghost planes on the other axes too (ghost_inner = 1); per axis, -1 = none
    int ghost_inner, ghost3_lo[3], ghost3_hi[3];
    // the box of cells [run_lo, run_hi) (per axis x, y, z) an AA step launch of
    // lbm_step_box / lbm_step_planes covers (read by the BOX kernels only)
    int run_lo[3], run_hi[3];
    // AA step launches over rows that are not a multiple of 32 cells (linear = 1): one thread
    // per cell in storage order, so that no thread idles past the end of a row and every warp
    // covers 32 consecutive cells; the coordinates come from dividing by nx
    int linear;
    Divisor div_nx;
    int box_lo[3], box_hi[3];  // solid cells' box widened by one (inclusive; empty: lo > hi)
    int face_dir[6];       // per face: 1 = Dirichlet wall (thermal)
    float T_wall[6];
    // immersed boundary: per-cell force (3 planes of S, consumed and zeroed by the step),
    // samples as planes of ib_cap: position (3), boundary velocity (3), weight, penalty (3)
    float *fib;
    const float *ibx, *ibub, *ibw;
    float *ibg;
    int ib_n, ib_cap;
    // bounding box of the samples' stencil cells, kept on the device by the marking kernel:
    // {-lo_x, -lo_y, -lo_z, hi_x, hi_y, hi_z} (all very negative when there is no sample)
    const int *ib_box;
};

// Neighbour offsets with periodic wrap by compare and add.
struct Offs {
    int xp, xm, yp, ym, zp, zm;
};

LBM_HD Offs make_offs(int x, int y, int z, const Params &P)
{
    Offs o;
    const int sy = P.nx, sz = P.nx * P.ny;
    o.xp = (x == P.nx - 1) ? 1 - P.nx : 1;
    o.xm = (x == 0) ? P.nx - 1 : -1;
    o.yp = (y == P.ny - 1) ? (1 - P.ny) * sy : sy;
    o.ym = (y == 0) ? (P.ny - 1) * sy : -sy;
    o.zp = (z == P.nz - 1) ? (1 - P.nz) * sz : sz;
    o.zm = (z == 0) ? (P.nz - 1) * sz : -sz;
    return o;
}

// Offset of the cell at x + (cx, cy, cz) (constants after unrolling).
LBM_HD int nb(const Offs &o, int cx, int cy, int cz)
{
    return (cx > 0 ? o.xp : cx < 0 ? o.xm : 0) + (cy > 0 ? o.yp : cy < 0 ? o.ym : 0) +
           (cz > 0 ? o.zp : cz < 0 ? o.zm : 0);
}

LBM_HD bool bit(uint32_t m, int b) { return (m >> b) & 1u; }

// A cell on a ghost plane of a slab (outer axis: z in 3-D, y in 2-D) or of a block (any
// axis).  Masked kernels see GHOST_BIT; unmasked ones (neither walls nor solids) test the
// coordinates: the outer axis always, the others only in blocks (a uniform flag).
template <class L>
LBM_HD bool ghost_plane(const Params &P, int x, int y, int z)
{
    const int c = L::DIM == 3 ? z : y;
    if (c == P.ghost_lo || c == P.ghost_hi) return true;
    if (!P.ghost_inner) return false;
    return x == P.ghost3_lo[0] || x == P.ghost3_hi[0] || y == P.ghost3_lo[1] ||
           y == P.ghost3_hi[1] || (L::DIM == 3 && (z == P.ghost3_lo[2] || z == P.ghost3_hi[2]));
}

// ---------------------------------------------------------------- cell access ---------

// Element index of slot (q, cell): 32-bit (NARROW) when every index of the population
// arrays fits in 32 bits, which keeps the address arithmetic of the 19 + 7 accesses in
// single registers; 64-bit otherwise.
template <bool NARROW>
LBM_HD auto slot(const Params &P, int q, int cell)
{
    if constexpr (NARROW) return (unsigned)q * (unsigned)P.S + (unsigned)cell;
    else return (size_t)q * P.S + (size_t)(unsigned)cell;
}

// Read patterns of the logical state (population q of cell x at the current time):
//   NATURAL  (q, x): after an even number of AA steps; the SPLIT mode.
//   AA_ODD   (opp q, x - c_q), or (q, x) on a wall link: after an odd number of AA steps.
//   PULL     (q, x - c_q), or (opp q, x) on a wall link: the PULL mode (post-collision state).
// On a wall link (the link x -> x - c_q, i.e. mask bit opp q) the stored value is the cell's
// own post-collision f_opp(q); for a Dirichlet thermal link it is turned into the
// anti-bounce-back value omega T_w - g.
enum { NATURAL = 0, AA_ODD = 1, PULL = 2 };

// Load the logical populations of a fluid cell with read pattern PAT.
template <class L, class TL, bool MASKED, int PAT, bool NARROW = false>
LBM_HD void load_cell(const Params &P, int idx, const Offs &o, uint32_t m, float (&f)[L::Q],
                      float (&g)[TL::QA])
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        if (PAT == NATURAL || q == 0) {
            f[q] = P.f[slot<NARROW>(P, q, idx)];
        } else {
            const int oq = L::opp(q);
            const bool wall_in = MASKED && bit(m, oq);
            const int own = PAT == AA_ODD ? q : oq, far = PAT == AA_ODD ? oq : q;
            f[q] = P.f[wall_in ? slot<NARROW>(P, own, idx)
                               : slot<NARROW>(P, far, idx + nb(o, -L::cx(q), -L::cy(q), -L::cz(q)))];
        }
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) {
            if (PAT == NATURAL || k == 0) {
                g[k] = P.g[slot<NARROW>(P, k, idx)];
            } else {
                const int ok = L::opp(k);
                const bool wall_in = MASKED && bit(m, ok);
                const int own = PAT == AA_ODD ? k : ok, far = PAT == AA_ODD ? ok : k;
                if (wall_in) {
                    const float raw = P.g[slot<NARROW>(P, own, idx)];
                    g[k] = bit(m, DIRICHLET_SHIFT + ok) ? P.abbT[ok] - raw : raw;
                } else {
                    g[k] = P.g[slot<NARROW>(P, far, idx + nb(o, -L::cx(k), -L::cy(k), -L::cz(k)))];
                }
            }
        }
    }
}

// After load_cell<..., MASKED=false, PAT> loaded every population as if no link were a
// wall (so that all loads issue without waiting for the mask), replace the ones whose
// link is a wall by the cell's own slot.  Only cells next to a wall or a solid take this
// branch; the speculative loads they discard read valid slots of other cells.
template <class L, class TL, int PAT, bool NARROW>
LBM_HD void fix_wall_loads(const Params &P, int idx, uint32_t m, float (&f)[L::Q],
                           float (&g)[TL::QA])
{
    static_assert(PAT != NATURAL, "natural reads have no wall redirect");
#pragma unroll
    for (int q = 1; q < L::Q; ++q) {
        const int oq = L::opp(q);
        if (bit(m, oq)) f[q] = P.f[slot<NARROW>(P, PAT == AA_ODD ? q : oq, idx)];
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 1; k < TL::Q; ++k) {
            const int ok = L::opp(k);
            if (bit(m, ok)) {
                const float raw = P.g[slot<NARROW>(P, PAT == AA_ODD ? k : ok, idx)];
                g[k] = bit(m, DIRICHLET_SHIFT + ok) ? P.abbT[ok] - raw : raw;
            }
        }
    }
}

template <class L>
LBM_HD constexpr uint32_t wall_bits() { return (1u << L::Q) - 2u; }

// Mask bits of the links with c_x = SIGN (the links that leave through the -x face when
// SIGN = -1, through the +x face when SIGN = +1).
template <class L, int SIGN>
LBM_HD constexpr uint32_t x_links()
{
    uint32_t b = 0;
    for (int q = 1; q < L::Q; ++q)
        if (L::cx(q) == SIGN) b |= 1u << q;
    return b;
}

// The wall links of cell x that the coordinates alone decide: those through an x face that
// is a wall.  With walls on x every row of cells has one such cell at each end, so the
// first and last warp of each row would otherwise wait for the mask before loading them.
template <class L>
LBM_HD uint32_t x_wall_links(const Params &P, int x)
{
    uint32_t b = 0;
    if (x == 0 && P.face_wall[0]) b |= x_links<L, -1>();
    if (x == P.nx - 1 && P.face_wall[1]) b |= x_links<L, +1>();
    return b;
}

// Mask bits of the links with c_a = SIGN along axis a, and the Dirichlet bits of the
// thermal links among them (thermal link k is flow link k, an axis link).
template <class L, int A, int SIGN>
LBM_HD constexpr uint32_t axis_links()
{
    uint32_t b = 0;
    for (int q = 1; q < L::Q; ++q) {
        const int c = A == 0 ? L::cx(q) : A == 1 ? L::cy(q) : L::cz(q);
        if (c == SIGN) b |= 1u << q;
    }
    return b;
}

template <class L, class TL, int A, int SIGN>
LBM_HD constexpr uint32_t axis_dirichlet()
{
    uint32_t b = 0;
    for (int k = 1; k < TL::Q; ++k) {
        const int c = A == 0 ? L::cx(k) : A == 1 ? L::cy(k) : L::cz(k);
        if (c == SIGN) b |= 1u << (DIRICHLET_SHIFT + k);
    }
    return b;
}

// Faces of axis A that cell coordinate c touches, as mask bits (wall links, and the
// Dirichlet bits of the thermal links through Dirichlet faces).
template <class L, class TL, int A>
LBM_HD uint32_t face_bits(const Params &P, int c, int n)
{
    uint32_t m = 0;
    if (c == 0 && P.face_wall[2 * A])
        m |= axis_links<L, A, -1>() | (P.face_dir[2 * A] ? axis_dirichlet<L, TL, A, -1>() : 0u);
    if (c == n - 1 && P.face_wall[2 * A + 1])
        m |= axis_links<L, A, +1>() | (P.face_dir[2 * A + 1] ? axis_dirichlet<L, TL, A, +1>() : 0u);
    return m;
}

// The link mask of a cell that neither is solid nor has a link into a solid cell: cell_mask
// from the face kinds alone, for every cell that is not on a slab's ghost plane.
// A link is a wall link when it leaves through a wall face along any axis; a thermal link
// crosses one face only.
template <class L, class TL>
LBM_HD uint32_t face_mask(const Params &P, int x, int y, int z)
{
    uint32_t m = face_bits<L, TL, 0>(P, x, P.nx) | face_bits<L, TL, 1>(P, y, P.ny);
    if constexpr (L::DIM == 3) m |= face_bits<L, TL, 2>(P, z, P.nz);
    return m;
}

// The link mask of a cell for the AA step kernels: loaded inside the box around the solid
// cells, the face bits elsewhere (no cell outside the box is solid or has a link into a
// solid cell).  IB: also loaded inside the box around the immersed-boundary samples'
// stencil cells (the only cells with IB_BIT).
template <class L, class TL, bool IB = false>
LBM_HD uint32_t boxed_mask(const Params &P, int idx, int x, int y, int z)
{
    bool inside = x >= P.box_lo[0] && x <= P.box_hi[0] && y >= P.box_lo[1] &&
                  y <= P.box_hi[1] && z >= P.box_lo[2] && z <= P.box_hi[2];
    if constexpr (IB) {
        const int *b = P.ib_box;
        inside = inside || (x >= -b[0] && y >= -b[1] && z >= -b[2] && x <= b[3] && y <= b[4] &&
                            z <= b[5]);
    }
    return inside ? P.mask[idx] : face_mask<L, TL>(P, x, y, z);
}

// Odd-step load (read pattern AA_ODD) that redirects the links in xw, a subset of
// x_wall_links, to the cell's own slots, as load_cell does for every wall link, and loads
// all other links from the neighbours.  Thermal values are the raw stored ones: the
// anti-bounce-back sign flip and omega T_w need the mask (abb_x_links).
template <class L, class TL, bool NARROW>
LBM_HD void load_odd_xwall(const Params &P, int idx, const Offs &o, uint32_t xw,
                           float (&f)[L::Q], float (&g)[TL::QA])
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        if (q == 0) {
            f[q] = P.f[slot<NARROW>(P, 0, idx)];
            continue;
        }
        const int oq = L::opp(q);
        const bool wall_in = L::cx(q) != 0 && bit(xw, oq);
        f[q] = P.f[wall_in ? slot<NARROW>(P, q, idx)
                           : slot<NARROW>(P, oq, idx + nb(o, -L::cx(q), -L::cy(q), -L::cz(q)))];
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) {
            if (k == 0) {
                g[k] = P.g[slot<NARROW>(P, 0, idx)];
                continue;
            }
            const int ok = L::opp(k);
            const bool wall_in = L::cx(k) != 0 && bit(xw, ok);
            g[k] = P.g[wall_in ? slot<NARROW>(P, k, idx)
                               : slot<NARROW>(P, ok, idx + nb(o, -L::cx(k), -L::cy(k), -L::cz(k)))];
        }
    }
}

// Anti-bounce-back on the thermal links loaded by load_odd_xwall from the own slot, once
// the mask (with its Dirichlet bits) is in.
template <class L, class TL>
LBM_HD void abb_x_links(const Params &P, uint32_t m, uint32_t xw, float (&g)[TL::QA])
{
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 1; k < TL::Q; ++k) {
            const int ok = L::opp(k);
            if (L::cx(k) != 0 && bit(xw, ok) && bit(m, DIRICHLET_SHIFT + ok))
                g[k] = P.abbT[ok] - g[k];
        }
    }
}

// Store populations into the natural slots (q, x) of the given arrays.
template <class L, class TL, bool NARROW>
LBM_HD void store_natural(const Params &P, float *F, float *G, int idx, const float (&f)[L::Q],
                          const float (&g)[TL::QA])
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q) F[slot<NARROW>(P, q, idx)] = f[q];
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) G[slot<NARROW>(P, k, idx)] = g[k];
    }
}

// Store post-collision populations.  Even: swapped into (opp q, x).  Odd: to (q, x + c_q)
// or, for a wall link, to (opp q, x) with bounce-back / anti-bounce-back applied.
template <class L, class TL, bool MASKED, bool ODD, bool NARROW = false>
LBM_HD void store_cell(const Params &P, int idx, const Offs &o, uint32_t m,
                       const float (&f)[L::Q], const float (&g)[TL::QA])
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        const int oq = L::opp(q);
        if (!ODD) {
            P.f[slot<NARROW>(P, oq, idx)] = f[q];
        } else if (q == 0) {
            P.f[slot<NARROW>(P, 0, idx)] = f[0];
        } else {
            const bool wall_out = MASKED && bit(m, q);
            P.f[wall_out ? slot<NARROW>(P, oq, idx)
                         : slot<NARROW>(P, q, idx + nb(o, L::cx(q), L::cy(q), L::cz(q)))] = f[q];
        }
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) {
            const int ok = L::opp(k);
            if (!ODD) {
                P.g[slot<NARROW>(P, ok, idx)] = g[k];
            } else if (k == 0) {
                P.g[slot<NARROW>(P, 0, idx)] = g[0];
            } else {
                const bool wall_out = MASKED && bit(m, k);
                if (wall_out) {
                    P.g[slot<NARROW>(P, ok, idx)] =
                        bit(m, DIRICHLET_SHIFT + k) ? P.abbT[k] - g[k] : g[k];
                } else {
                    P.g[slot<NARROW>(P, k, idx + nb(o, L::cx(k), L::cy(k), L::cz(k)))] = g[k];
                }
            }
        }
    }
}

// Store logical populations so that load_cell<..., PAT> reads them back (initialisation
// and set_populations; the inverse of load_cell).
template <class L, class TL, bool MASKED, int PAT>
LBM_HD void store_logical(const Params &P, int idx, const Offs &o, uint32_t m,
                          const float (&f)[L::Q], const float (&g)[TL::QA])
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        if (PAT == NATURAL || q == 0) {
            P.f[slot<false>(P, q, idx)] = f[q];
        } else {
            const int oq = L::opp(q);
            const bool wall_in = MASKED && bit(m, oq);
            const int own = PAT == AA_ODD ? q : oq, far = PAT == AA_ODD ? oq : q;
            P.f[wall_in ? slot<false>(P, own, idx)
                        : slot<false>(P, far, idx + nb(o, -L::cx(q), -L::cy(q), -L::cz(q)))] = f[q];
        }
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) {
            if (PAT == NATURAL || k == 0) {
                P.g[slot<false>(P, k, idx)] = g[k];
            } else {
                const int ok = L::opp(k);
                const int own = PAT == AA_ODD ? k : ok, far = PAT == AA_ODD ? ok : k;
                if (MASKED && bit(m, ok)) {
                    P.g[slot<false>(P, own, idx)] =
                        bit(m, DIRICHLET_SHIFT + ok) ? P.abbT[ok] - g[k] : g[k];
                } else {
                    P.g[slot<false>(P, far, idx + nb(o, -L::cx(k), -L::cy(k), -L::cz(k)))] = g[k];
                }
            }
        }
    }
}

// ------------------------------------------------------------------ the step ----------

// Programmatic dependent launch (sm_90 and later).  A kernel launched with programmatic
// stream serialization (launch_chained) may be scheduled while the kernel before it in the
// stream is still running; before it touches anything that kernel wrote it waits
// (griddepcontrol.wait) until that kernel has completed and its writes are visible.
// allow_dependents lets the next such kernel be scheduled once every block of this one has
// started, so that its blocks fill the SMs freed during this kernel's last wave instead of
// after it.  Both are no-ops in a kernel launched without the attribute, and on the host.
LBM_HD void allow_dependents()
{
#if defined(__CUDA_ARCH__)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

LBM_HD void wait_prerequisites()
{
#if defined(__CUDA_ARCH__)
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Read the immersed-boundary force of a cell and zero it for the next step: one atomic
// exchange per component on the device.  Measured on GB300 (128^3 channel, 12,868 samples),
// a plain load followed by a store of these values (accumulated by the immersed-boundary
// kernel's atomic additions just before, a few lanes per warp) slowed every block on the
// GPU while the planes holding stencil cells were stepped, about 7 us of a 66 us step; the
// exchange costs about 0.3 us.  (The step's own loads and stores of the populations, at the
// same addresses in every cell, show no such cost.)  The host emulation runs one thread:
// there a load and a store do.
LBM_HD void take_ib_force(const Params &P, int idx, float (&ext)[3])
{
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        float *p = P.fib + ((size_t)a * P.S + (unsigned)idx);
#if defined(__CUDA_ARCH__)
        ext[a] = atomicExch(p, 0.0f);
#else
        ext[a] = *p;
        *p = 0.0f;
#endif
    }
}

// One AA step of cell (x, y, z): loads through Pr, stores through Pw (the same buffer in
// the kernel; a separate one in the host emulation of the tests).
// IB: the context has immersed-boundary samples (cells with IB_BIT take a per-cell force);
// kernels without it carry no trace of that path.
// FACES (with MASKED): the mask comes from the coordinates (face_mask) outside the box of
// the solid cells (and, with IB, of the samples' stencil cells) and is loaded only inside
// it (boxed_mask).
template <class L, class TL, int COLL, bool MASKED, bool ODD, bool NARROW, bool IB = false,
          bool FACES = false>
LBM_HD void aa_step_cell(const Params &Pr, const Params &Pw, int x, int y, int z)
{
    static_assert(!FACES || MASKED, "FACES is a masked form");
    if ((!MASKED || FACES) && ghost_plane<L>(Pr, x, y, z)) return;
    const int idx = x + Pr.nx * (y + Pr.ny * z);
    // The mask load and the population loads are issued together: the populations are
    // loaded as if no link were a wall (except the x-face wall links, known from x), and
    // the remaining wall links are fixed once the mask is in.
    const uint32_t m = FACES ? boxed_mask<L, TL, IB>(Pr, idx, x, y, z) : MASKED ? Pr.mask[idx] : 0u;
    float f[L::Q], g[TL::QA];
    // wall links through an x face need no mask: they are redirected at once
    const uint32_t xw = (MASKED && ODD) ? x_wall_links<L>(Pr, x) : 0u;
    {
        Offs o{};
        if (ODD) o = make_offs(x, y, z, Pr);
        if (MASKED && ODD)
            load_odd_xwall<L, TL, NARROW>(Pr, idx, o, xw, f, g);
        else
            load_cell<L, TL, false, ODD ? AA_ODD : NATURAL, NARROW>(Pr, idx, o, 0u, f, g);
    }
    float ext[3];
    if (MASKED) {
        if (m & SKIP_BITS) return;
        if (ODD) {
            const uint32_t rest = m & ~xw;   // Dirichlet bits stay; x-face links are done
            if (rest & wall_bits<L>()) fix_wall_loads<L, TL, AA_ODD, NARROW>(Pr, idx, rest, f, g);
            if (xw) abb_x_links<L, TL>(Pr, m, xw, g);
        }
    }
    if constexpr (IB) {
        const bool forced = m & IB_BIT;
        if (forced) take_ib_force(Pr, idx, ext);
        collide<L, TL, COLL>(f, g, Pr.c, forced ? ext : nullptr);
    } else {
        (void)ext;
        collide<L, TL, COLL>(f, g, Pr.c);
    }
    // Recompute the store addresses after the collision instead of keeping the load-time
    // values live through it (the empty asm hides that they are the same).
    int xs = x, ys = y, zs = z, is = idx;
    uint32_t ms = m;
    asm volatile("" : "+r"(xs), "+r"(ys), "+r"(zs), "+r"(is), "+r"(ms));
    Offs o{};
    if (ODD) o = make_offs(xs, ys, zs, Pw);
    if constexpr (MASKED && ODD) {
        // only cells next to a wall or solid redirect stores; the rest (whole warps away
        // from the walls) take the plain neighbour stores
        if (ms & wall_bits<L>()) store_cell<L, TL, true, true, NARROW>(Pw, is, o, ms, f, g);
        else store_cell<L, TL, false, true, NARROW>(Pw, is, o, 0u, f, g);
    } else {
        store_cell<L, TL, MASKED, ODD, NARROW>(Pw, is, o, ms, f, g);
    }
}

// Cell t of a linear AA step launch over whole planes of the outer axis: in 3-D, cell t of
// plane `plane` of the launch in storage order; in 2-D, cell t of the launch's rows.  BOX:
// the launch starts at plane P.run_lo[2] (3-D) or row P.run_lo[1] (2-D) and, in 2-D, ends
// at row P.run_hi[1]; otherwise it covers the whole grid.  false past the plane (3-D) or
// past the launch's last row (2-D).
template <class L, bool BOX>
LBM_HD bool linear_cell_coords(const Params &P, int t, int plane, int &x, int &y, int &z)
{
    if constexpr (L::DIM == 3) {
        if (t >= P.nx * P.ny) return false;
        z = BOX ? P.run_lo[2] + plane : plane;
        y = (int)div_by((unsigned)t, P.div_nx);
        x = t - y * P.nx;
    } else {
        const int i = BOX ? P.run_lo[1] * P.nx + t : t;
        if (i >= (BOX ? P.run_hi[1] : P.ny) * P.nx) return false;
        y = (int)div_by((unsigned)i, P.div_nx);
        x = i - y * P.nx;
        z = 0;
    }
    return true;
}

// Cell of the calling thread in an AA step launch: blocks along x, rows stacked in y,
// planes in z (3-D); or, with P.linear, a grid over the cells of whole planes in storage
// order.  BOX (lbm_step_box): the launch covers the box [P.run_lo, P.run_hi) and is offset
// by run_lo; otherwise the whole grid, with no offset at all (the plain steps keep the
// simplest index arithmetic).  Returns false for threads past the launch's edge.
template <class L, bool BOX>
LBM_HD bool step_cell_coords(const Params &P, int &x, int &y, int &z)
{
#if defined(__CUDA_ARCH__)
    if (P.linear)
        return linear_cell_coords<L, BOX>(P, blockIdx.x * blockDim.x + threadIdx.x, blockIdx.y,
                                          x, y, z);
    x = blockIdx.x * blockDim.x + threadIdx.x;
    y = blockIdx.y * blockDim.y + threadIdx.y;
    z = blockIdx.z;
#endif
    if constexpr (BOX) {
        x += P.run_lo[0];
        y += P.run_lo[1];
        z += P.run_lo[2];
        return x < P.run_hi[0] && y < P.run_hi[1];
    } else {
        return x < P.nx && y < P.ny;
    }
}

// Whether cell (x, y, z) lies within two cells of the box of the immersed-boundary samples'
// stencil cells (P.ib_box), along periodic wraps too.  The step on a cell farther away
// touches no slot the immersed-boundary kernel reads and needs none of its forces.
template <class L>
LBM_HD bool near_ib_box(const Params &P, int x, int y, int z)
{
    const int c[3] = {x, y, z}, n[3] = {P.nx, P.ny, P.nz};
    for (int a = 0; a < L::DIM; ++a) {
        const int lo = -P.ib_box[a] - 2, hi = P.ib_box[3 + a] + 2;
        if (hi < lo) return false;                  // no sample
        if (hi - lo + 1 >= n[a]) continue;          // the whole axis
        int d = c[a] - lo;                          // distance above lo, modulo n
        if (d < 0) d += n[a];
        else if (d >= n[a]) d -= n[a];
        if (d > hi - lo) return false;
    }
    return true;
}

// The start of a step launch: the cell of the calling thread, and the wait for the kernel
// before it (every load reads the previous step's stores).  With immersed-boundary samples
// (IB and P.ib_n > 0) the kernel before is the immersed-boundary kernel, which releases
// this launch only once the previous step has completed (it triggers its dependents after
// its own wait): then only cells near the samples wait for its forces, and the others start
// at once, beside it.
template <class L, bool IB, bool BOX>
LBM_HD bool step_start(const Params &P, int &x, int &y, int &z)
{
    if constexpr (!IB) {
        wait_prerequisites();
        return step_cell_coords<L, BOX>(P, x, y, z);
    } else {
        const bool in = step_cell_coords<L, BOX>(P, x, y, z);
        if (P.ib_n == 0 || !in || near_ib_box<L>(P, x, y, z)) wait_prerequisites();
        return in;
    }
}

// One time step: one thread per cell, blocks along x (x fastest for coalescing).
template <class L, class TL, int COLL, bool MASKED, bool ODD, bool NARROW, bool IB,
          bool FACES = false, bool BOX = false>
__global__ void __launch_bounds__(256) step_kernel(const Params P)
{
    allow_dependents();
    int x = 0, y = 0, z = 0;
    if (!step_start<L, IB, BOX>(P, x, y, z)) return;
    aa_step_cell<L, TL, COLL, MASKED, ODD, NARROW, IB, FACES>(P, P, x, y, z);
}

// The same step with the register allocation bounded so that 5 blocks of 256 reside per SM
// (48 registers): for a collision long enough that the extra warps pay for themselves.
template <class L, class TL, int COLL, bool MASKED, bool ODD, bool NARROW, bool IB,
          bool FACES = false, bool BOX = false>
__global__ void __launch_bounds__(256, 5) step_kernel_5(const Params P)
{
    allow_dependents();
    int x = 0, y = 0, z = 0;
    if (!step_start<L, IB, BOX>(P, x, y, z)) return;
    aa_step_cell<L, TL, COLL, MASKED, ODD, NARROW, IB, FACES>(P, P, x, y, z);
}

// Two-buffer PULL step: pull from the current buffer, collide, write the other buffer's
// natural slots.  No slot is read and written in the same launch.
template <class L, class TL, int COLL, bool MASKED, bool NARROW, bool IB = false>
LBM_HD void pull_step_cell(const Params &P, float *Wf, float *Wg, int x, int y, int z)
{
    const int idx = x + P.nx * (y + P.ny * z);
    const uint32_t m = MASKED ? P.mask[idx] : 0u;
    float f[L::Q], g[TL::QA];
    {
        const Offs o = make_offs(x, y, z, P);
        load_cell<L, TL, false, PULL, NARROW>(P, idx, o, 0u, f, g);
    }
    float ext[3];
    if (MASKED) {
        if (m & SKIP_BITS) return;
        if (m & wall_bits<L>()) fix_wall_loads<L, TL, PULL, NARROW>(P, idx, m, f, g);
    }
    if constexpr (IB) {
        const bool forced = m & IB_BIT;
        if (forced) take_ib_force(P, idx, ext);
        collide<L, TL, COLL>(f, g, P.c, forced ? ext : nullptr);
    } else {
        (void)ext;
        collide<L, TL, COLL>(f, g, P.c);
    }
    int is = idx;
    asm volatile("" : "+r"(is));
    store_natural<L, TL, NARROW>(P, Wf, Wg, is, f, g);
}

template <class L, class TL, int COLL, bool MASKED, bool NARROW, bool IB>
__global__ void __launch_bounds__(256) pull_kernel(const Params P)
{
    allow_dependents();
    wait_prerequisites();
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    pull_step_cell<L, TL, COLL, MASKED, NARROW, IB>(P, P.fo, P.go, x, y, z);
}

// SPLIT mode, pass 1: collide cell idx in place in the natural slots.
template <class L, class TL, int COLL, bool MASKED, bool NARROW, bool IB = false>
LBM_HD void collide_in_place_cell(const Params &P, int idx)
{
    const uint32_t m = MASKED ? P.mask[idx] : 0u;
    if (m & SKIP_BITS) return;
    float f[L::Q], g[TL::QA], ext[3];
    const Offs o{};
    load_cell<L, TL, false, NATURAL, NARROW>(P, idx, o, 0u, f, g);
    if constexpr (IB) {
        const bool forced = m & IB_BIT;
        if (forced) take_ib_force(P, idx, ext);
        collide<L, TL, COLL>(f, g, P.c, forced ? ext : nullptr);
    } else {
        (void)ext;
        collide<L, TL, COLL>(f, g, P.c);
    }
    store_natural<L, TL, NARROW>(P, P.f, P.g, idx, f, g);
}

template <class L, class TL, int COLL, bool MASKED, bool NARROW, bool IB>
__global__ void __launch_bounds__(256) collide_kernel(const Params P)
{
    allow_dependents();
    wait_prerequisites();
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    collide_in_place_cell<L, TL, COLL, MASKED, NARROW, IB>(P, x + P.nx * (y + P.ny * z));
}

// SPLIT mode, pass 2: pull the post-collision populations of cell (x, y, z) into W.
template <class L, class TL, bool MASKED, bool NARROW>
LBM_HD void stream_cell(const Params &P, float *Wf, float *Wg, int x, int y, int z)
{
    const int idx = x + P.nx * (y + P.ny * z);
    uint32_t m = 0;
    if (MASKED) {
        m = P.mask[idx];
        if (m & SKIP_BITS) return;
    }
    float f[L::Q], g[TL::QA];
    const Offs o = make_offs(x, y, z, P);
    load_cell<L, TL, MASKED, PULL, NARROW>(P, idx, o, m, f, g);
    store_natural<L, TL, NARROW>(P, Wf, Wg, idx, f, g);
}

template <class L, class TL, bool MASKED, bool NARROW>
__global__ void __launch_bounds__(256) stream_kernel(const Params P)
{
    allow_dependents();
    wait_prerequisites();
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    stream_cell<L, TL, MASKED, NARROW>(P, P.fo, P.go, x, y, z);
}

// -------------------------------------------------------------- immersed boundary -----

// Immersed boundary ("GPU Optimization for High-Quality Kinetic Fluid Simulation", Sec. 3.1,
// Eq. 6-8).  Corner c (0 .. 2^dim - 1) of sample s's stencil: its cell, its trilinear weight
// K, and K rho, K u with rho and u = (j + F_body/2)/rho of the logical state (read with
// pattern PAT).  A solid stencil cell counts as rho = 1, u = 0.  Sample positions were
// checked on the host: stencils never leave through a wall face.
// The cell (returned) of corner c of sample s's stencil and its weight K; q receives its
// coordinates.
template <class L>
LBM_HD int ib_corner_cell(const Params &P, int s, int c, float &K, int (&q)[3])
{
    const int dim = L::DIM;
    const int n[3] = {P.nx, P.ny, P.nz};
    q[0] = q[1] = q[2] = 0;
    float k = 1.0f;
    for (int a = 0; a < dim; ++a) {
        const float xa = P.ibx[a * P.ib_cap + s];
        const int base = (int)floorf(xa);
        const float fr = xa - (float)base;
        const int d = (c >> a) & 1;
        q[a] = base + d;
        if (q[a] >= n[a]) q[a] -= n[a];
        k *= d ? fr : 1.0f - fr;
    }
    K = k;
    return q[0] + P.nx * (q[1] + P.ny * q[2]);
}

// K rho and K u of the corner cell idx (coordinates q, link mask m) of weight k.
template <class L, class TL, int PAT>
LBM_HD void ib_corner_moments(const Params &P, int idx, const int (&q)[3], float k, uint32_t m,
                              float &Krho, float (&Ku)[3])
{
    // the populations load as if no link were a wall; wall links are fixed after
    Offs o{};
    if (PAT != NATURAL) o = make_offs(q[0], q[1], q[2], P);
    float f[L::Q], g[TL::QA];
    load_cell<L, TL, false, PAT>(P, idx, o, 0u, f, g);
    if (m & SOLID_BIT) {
        Krho = k;
        Ku[0] = Ku[1] = Ku[2] = 0.0f;
        return;
    }
    if constexpr (PAT != NATURAL) {
        if (m & wall_bits<L>()) fix_wall_loads<L, TL, PAT, false>(P, idx, m, f, g);
    }
    float dr = 0.0f, jx = 0.0f, jy = 0.0f, jz = 0.0f, t = 0.0f;
    for (int i = 0; i < L::Q; ++i) {
        dr += f[i];
        jx += L::cx(i) * f[i];
        jy += L::cy(i) * f[i];
        jz += L::cz(i) * f[i];
    }
    if constexpr (TL::Q > 0) {
        for (int i = 0; i < TL::Q; ++i) t += g[i];
    }
    const float r = 1.0f + dr;
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<(TL::Q > 0)>(P.c, r, t, jx, jy, jz, Fx, Fy, Fz, ux, uy, uz);
    Krho = k * r;
    Ku[0] = k * ux;
    Ku[1] = k * uy;
    Ku[2] = k * uz;
}

template <class L, class TL, int PAT>
LBM_HD int ib_corner(const Params &P, int s, int c, float &K, float &Krho, float (&Ku)[3])
{
    int q[3];
    const int idx = ib_corner_cell<L>(P, s, c, K, q);
    ib_corner_moments<L, TL, PAT>(P, idx, q, K, P.mask ? P.mask[idx] : 0u, Krho, Ku);
    return idx;
}

// Sample order ("GPU Optimization for High-Quality Kinetic Fluid Simulation", Sec. 4,
// Fig. 7): samples sorted by the l x l x l block of the grid they lie in (blocks in x-y-z
// order), then by the Morton code of their position inside the block (8 bits per axis),
// so that the samples one warp handles touch nearby cells.
constexpr int IB_MORTON_BITS = 24;

// Spread the low 8 bits of v to every third bit (Morton interleave).
LBM_HD uint32_t spread3(uint32_t v)
{
    v &= 0xffu;
    v = (v | (v << 8)) & 0x0000f00fu;
    v = (v | (v << 4)) & 0x000c30c3u;
    v = (v | (v << 2)) & 0x00249249u;
    return v;
}

// Sort key of a sample at (wrapped, checked) position x: (block index << 24) | Morton code.
// nbx, nby: blocks along x and y.  The host and the device compute it with the same fp32
// operations, so both order samples identically.
LBM_HD unsigned long long ib_sort_key(const float (&x)[3], int dim, int l, long long nbx,
                                      long long nby)
{
    long long b[3] = {0, 0, 0};
    uint32_t m = 0;
    for (int a = 0; a < dim; ++a) {
        const float v = x[a];
        b[a] = (long long)(v / (float)l);
        const float in = v - (float)(b[a] * l);
        float t = in * (256.0f / (float)l);
        t = t < 255.0f ? t : 255.0f;
        m |= spread3(t > 0.0f ? (uint32_t)t : 0u) << a;
    }
    const unsigned long long block = (unsigned long long)(b[0] + nbx * (b[1] + nby * b[2]));
    return (block << IB_MORTON_BITS) | m;
}

// Position of a sample given in cells: periodic axes wrap into [0, n); on a wall axis the
// stencil (base and base + 1) must stay inside, i.e. 0 <= x < n - 1.  Returns false for a
// non-finite position or a stencil that would leave through a wall face.
LBM_HD bool ib_place(const Params &P, int dim, const float *in, float (&x)[3])
{
    const int ext[3] = {P.nx, P.ny, P.nz};
    bool ok = true;
    for (int a = 0; a < 3; ++a) {
        float v = a < dim ? in[a] : 0.0f;
        if (!(fabsf(v) <= 3.402823466e38f)) {   // NaN or infinite
            ok = false;
            v = 0.0f;
        } else if (a < dim && !P.face_wall[2 * a]) {
            v = fmodf(v, (float)ext[a]);
            if (v < 0.0f) v += (float)ext[a];
            if (v >= (float)ext[a]) v = 0.0f;
        } else if (a < dim && !(v >= 0.0f && v < (float)(ext[a] - 1))) {
            ok = false;
        }
        x[a] = v;
    }
    return ok;
}

// Penalty from a sample's weight w, boundary velocity u_b and interpolated rho and u:
// g = w rho (u_b - u).
template <class L>
LBM_HD void ib_penalty(float w, const float (&ub)[3], float rho, const float (&u)[3],
                       float (&gs)[3])
{
    for (int a = 0; a < 3; ++a) gs[a] = (a < L::DIM) ? w * rho * (ub[a] - u[a]) : 0.0f;
}

// The same for sample s of the parameter block.
template <class L>
LBM_HD void ib_penalty(const Params &P, int s, float rho, const float (&u)[3], float (&gs)[3])
{
    const float ub[3] = {P.ibub[s], P.ibub[P.ib_cap + s], P.ibub[2 * P.ib_cap + s]};
    ib_penalty<L>(P.ibw[s], ub, rho, u, gs);
}

// Whole sample s, corner by corner (the host emulation's form of the kernel below).
template <class L, class TL, int PAT>
LBM_HD int ib_sample(const Params &P, int s, int (&node)[8], float (&K)[8], float (&gs)[3])
{
    const int corners = 1 << L::DIM;
    float rho = 0.0f, u[3] = {0.0f, 0.0f, 0.0f};
    for (int c = 0; c < corners; ++c) {
        float kr, ku[3];
        node[c] = ib_corner<L, TL, PAT>(P, s, c, K[c], kr, ku);
        rho += kr;
        for (int a = 0; a < 3; ++a) u[a] += ku[a];
    }
    ib_penalty<L>(P, s, rho, u, gs);
    return corners;
}

// One thread per stencil corner (2^dim threads per sample, adjacent lanes): each loads its
// cell, the group sums K rho and K u with shuffles, every thread forms the penalty and
// spreads its share K g into its cell with atomic additions (cells are shared between
// samples); corner 0 keeps the penalty for the diagnostics.  t: the corner's thread index
// over all samples; whole warps call this (the shuffles span 2^dim lanes).  Waits for the
// prerequisite grid (wait_prerequisites) before it reads any population.
template <class L, class TL, int PAT>
LBM_HD void ib_corner_thread(const Params &P, int t)
{
    constexpr int CORNERS = 1 << L::DIM;
    const int s = t / CORNERS, c = t % CORNERS;
    const bool active = s < P.ib_n;
    float K = 0.0f, kr = 0.0f, ku[3] = {0.0f, 0.0f, 0.0f};
    float w = 0.0f, ub[3] = {0.0f, 0.0f, 0.0f};
    int idx = 0, q[3] = {0, 0, 0};
    uint32_t m = 0;
    // The samples and the link mask are written only by the context's set-up and
    // sample-setting calls, which finish before the step before this kernel: read them,
    // and place the stencil, while that step is still running.
    if (active) {
        w = P.ibw[s];
        for (int a = 0; a < 3; ++a) ub[a] = P.ibub[a * P.ib_cap + s];
        idx = ib_corner_cell<L>(P, s, c, K, q);
        m = P.mask[idx];
    }
    wait_prerequisites();   // the stencil cells hold the previous step's stores
    // only now may the step after this kernel start: its cells away from the samples skip
    // their wait, and must find the previous step complete
    allow_dependents();
    if (active) ib_corner_moments<L, TL, PAT>(P, idx, q, K, m, kr, ku);
#if defined(__CUDA_ARCH__)
#pragma unroll
    for (int off = 1; off < CORNERS; off <<= 1) {
        kr += __shfl_xor_sync(0xffffffffu, kr, off, CORNERS);
        for (int a = 0; a < 3; ++a) ku[a] += __shfl_xor_sync(0xffffffffu, ku[a], off, CORNERS);
    }
    if (!active) return;
    float gs[3];
    ib_penalty<L>(w, ub, kr, ku, gs);
    if (c == 0)
        for (int a = 0; a < 3; ++a) P.ibg[a * P.ib_cap + s] = gs[a];
    if (m & SOLID_BIT) return;
    for (int a = 0; a < L::DIM; ++a)
        atomicAdd(P.fib + ((size_t)a * P.S + (unsigned)idx), K * gs[a]);
#endif
}

template <class L, class TL, int PAT>
__global__ void __launch_bounds__(128) ib_kernel(const Params P)
{
    ib_corner_thread<L, TL, PAT>(P, blockIdx.x * blockDim.x + threadIdx.x);
}

// Set (SET) or clear IB_BIT on the stencil cells of every sample of P: clearing the
// current samples' stencils before new samples replace them, then setting the new ones',
// keeps IB_BIT on exactly the stencil cells of the current samples.
// SET also grows box (the layout of Params::ib_box, reset beforehand) to cover the
// stencil cells: the step kernels load the mask inside it.
template <class L, bool SET>
__global__ void ib_mark_kernel(const Params P, uint32_t *mask, int *box)
{
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    const int dim = L::DIM;
    const int n[3] = {P.nx, P.ny, P.nz};
    int ext[6] = {INT_MIN, INT_MIN, INT_MIN, INT_MIN, INT_MIN, INT_MIN};   // -lo, hi
    if (s < P.ib_n) {
        int base[3] = {0, 0, 0};
        for (int a = 0; a < dim; ++a) base[a] = (int)floorf(P.ibx[a * P.ib_cap + s]);
        for (int c = 0; c < (1 << dim); ++c) {
            int q[3] = {base[0], base[1], base[2]};
            for (int a = 0; a < dim; ++a) {
                q[a] += (c >> a) & 1;
                if (q[a] >= n[a]) q[a] -= n[a];
            }
            for (int a = 0; a < 3; ++a) {
                ext[a] = max(ext[a], -q[a]);
                ext[3 + a] = max(ext[3 + a], q[a]);
            }
            uint32_t *m = mask + (q[0] + P.nx * (q[1] + P.ny * q[2]));
            if (SET) atomicOr(m, IB_BIT);
            else atomicAnd(m, ~IB_BIT);
        }
    }
    if (!SET) return;
    for (int k = 0; k < 6; ++k) {
        int v = ext[k];
        for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
        if ((threadIdx.x & 31) == 0 && v != INT_MIN) atomicMax(box + k, v);
    }
}

// ------------------------------------------------------------ auxiliary kernels -------

// f = f_eq(rho, u) - w, g = g_eq(T, u) as the logical state of one cell, stored for read
// pattern PAT (NATURAL for AA and SPLIT, PULL for the PULL mode).  f_eq is the quadratic
// equilibrium on D3Q19 / D2Q9 and the product form on D3Q27.
template <class L, class TL, int PAT = NATURAL>
LBM_HD void init_cell(const Params &P, int idx, const float *rho, const float *u,
                      const float *T, int x = 0, int y = 0, int z = 0)
{
    const size_t N = (size_t)P.nx * P.ny * P.nz;
    const bool solid = P.mask && (P.mask[idx] & SOLID_BIT);
    float f[L::Q], g[TL::QA];
    if (solid) {
#pragma unroll
        for (int q = 0; q < L::Q; ++q) f[q] = 0.0f;
#pragma unroll
        for (int k = 0; k < TL::QA; ++k) g[k] = 0.0f;
    } else {
        const float r = rho[idx];
        const float dr = r - 1.0f;
        const float ux = u[idx], uy = u[N + idx], uz = (L::DIM == 3) ? u[2 * N + idx] : 0.0f;
        if constexpr (L::Q == 27) {
#pragma unroll
            for (int q = 0; q < L::Q; ++q)
                f[q] = d3q27_feq_shifted(L::cx(q), L::cy(q), L::cz(q), dr, ux, uy, uz);
        } else {
            const float u15 = 1.5f * (ux * ux + uy * uy + uz * uz);
#pragma unroll
            for (int q = 0; q < L::Q; ++q) {
                const float cu = L::cx(q) * ux + L::cy(q) * uy + L::cz(q) * uz;
                f[q] = L::w(q) * (dr + r * (3.0f * cu + 4.5f * cu * cu - u15));
            }
        }
        if constexpr (TL::Q == 7) d3q7_equilibrium(g, P.c.a_T, T[idx], ux, uy, uz);
        if constexpr (TL::Q == 5) d2q5_equilibrium(g, P.c.a_T, T[idx], ux, uy);
    }
    if constexpr (PAT == NATURAL) {
        store_natural<L, TL, false>(P, P.f, P.g, idx, f, g);
    } else {
        if (solid) return;   // a solid cell's slots are never read
        const uint32_t m = P.mask ? P.mask[idx] : 0u;
        const Offs o = make_offs(x, y, z, P);
        store_logical<L, TL, true, PAT>(P, idx, o, m, f, g);
    }
}

template <class L, class TL, int PAT>
__global__ void init_kernel(const Params P, const float *__restrict__ rho,
                            const float *__restrict__ u, const float *__restrict__ T)
{
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    init_cell<L, TL, PAT>(P, x + P.nx * (y + P.ny * z), rho, u, T, x, y, z);
}

// Link mask of cell (x, y, z): bit q (1..Q-1) when the link x -> x + c_q leaves the
// domain through a WALL face or ends in a solid cell; bit 19 + k when thermal link k
// leaves through a Dirichlet face; bit 31 for a solid cell.
template <class L, class TL>
LBM_HD uint32_t cell_mask(const Params &P, const uint8_t *solid, int x, int y, int z)
{
    const int idx = x + P.nx * (y + P.ny * z);
    const int n[3] = {P.nx, P.ny, P.nz};
    const int c0[3] = {x, y, z};
    // halo planes of a slab: kept for the neighbours' slots, never updated
    uint32_t ghost = 0;
    for (int a = 0; a < 3; ++a)
        if ((P.face_halo[2 * a] && c0[a] == 0) || (P.face_halo[2 * a + 1] && c0[a] == n[a] - 1))
            ghost = GHOST_BIT;
    if (solid && solid[idx]) return SOLID_BIT | ghost;
    if (ghost) return ghost;
    uint32_t m = 0;
#pragma unroll
    for (int q = 1; q < L::Q; ++q) {
        const int c[3] = {L::cx(q), L::cy(q), L::cz(q)};
        int s[3];
        bool wall = false;
        int face = -1;
        for (int a = 0; a < 3; ++a) {
            s[a] = c0[a] + c[a];
            if (s[a] < 0) {
                if (P.face_wall[2 * a] || P.face_halo[2 * a]) { wall = true; face = 2 * a; }
                else s[a] += n[a];
            } else if (s[a] >= n[a]) {
                if (P.face_wall[2 * a + 1] || P.face_halo[2 * a + 1]) {
                    wall = true;
                    face = 2 * a + 1;
                }
                else s[a] -= n[a];
            }
        }
        if (!wall && solid && solid[s[0] + P.nx * (s[1] + P.ny * s[2])]) wall = true;
        if (wall) m |= 1u << q;
        if (TL::Q > 0 && q < TL::Q && face >= 0 && P.face_dir[face])
            m |= 1u << (DIRICHLET_SHIFT + q);
    }
    return m;
}

template <class L, class TL>
__global__ void mask_kernel(const Params P, const uint8_t *__restrict__ solid,
                            uint32_t *__restrict__ mask)
{
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    mask[x + P.nx * (y + P.ny * z)] = cell_mask<L, TL>(P, solid, x, y, z);
}

// Macroscopic fields of the logical state: rho, u = (j + F/2)/rho, T.
template <class L, class TL, bool MASKED, int PAT>
__global__ void macro_kernel(const Params P, float *__restrict__ rho, float *__restrict__ u,
                             float *__restrict__ T)
{
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    const int idx = x + P.nx * (y + P.ny * z);
    const size_t N = (size_t)P.nx * P.ny * P.nz;
    uint32_t m = 0;
    if (MASKED) m = P.mask[idx];
    if ((m & SKIP_BITS) || (!MASKED && ghost_plane<L>(P, x, y, z))) {
        if (rho) rho[idx] = 0.0f;
        if (u) {
            for (int a = 0; a < L::DIM; ++a) u[a * N + idx] = 0.0f;
        }
        if (T) T[idx] = 0.0f;
        return;
    }
    Offs o{};
    if (PAT != NATURAL) o = make_offs(x, y, z, P);
    float f[L::Q], g[TL::QA];
    load_cell<L, TL, MASKED, PAT>(P, idx, o, m, f, g);
    float dr = 0.0f, jx = 0.0f, jy = 0.0f, jz = 0.0f, t = 0.0f;
#pragma unroll
    for (int q = 0; q < L::Q; ++q) {
        dr += f[q];
        jx += L::cx(q) * f[q];
        jy += L::cy(q) * f[q];
        jz += L::cz(q) * f[q];
    }
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int k = 0; k < TL::Q; ++k) t += g[k];
    }
    const float r = 1.0f + dr;
    float Fx, Fy, Fz, ux, uy, uz;
    force_velocity<(TL::Q > 0)>(P.c, r, t, jx, jy, jz, Fx, Fy, Fz, ux, uy, uz);
    if (rho) rho[idx] = r;
    if (u) {
        u[idx] = ux;
        u[N + idx] = uy;
        if (L::DIM == 3) u[2 * N + idx] = uz;
    }
    if (T) T[idx] = t;
}

// Logical populations out (f unshifted), or in (SET).
template <class L, class TL, bool MASKED, int PAT, bool SET>
__global__ void pop_kernel(const Params P, float *__restrict__ fo, float *__restrict__ go)
{
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    const int z = blockIdx.z;
    if (x >= P.nx || y >= P.ny) return;
    const int idx = x + P.nx * (y + P.ny * z);
    const size_t N = (size_t)P.nx * P.ny * P.nz;
    uint32_t m = 0;
    if (MASKED) m = P.mask[idx];
    if ((m & SKIP_BITS) || (!MASKED && ghost_plane<L>(P, x, y, z))) {
        if (!SET) {
            for (int q = 0; q < L::Q; ++q) fo[q * N + idx] = 0.0f;
            if (TL::Q > 0 && go)
                for (int k = 0; k < TL::Q; ++k) go[k * N + idx] = 0.0f;
        }
        return;
    }
    Offs o{};
    if (PAT != NATURAL) o = make_offs(x, y, z, P);
    float f[L::Q], g[TL::QA];
    if (SET) {
#pragma unroll
        for (int q = 0; q < L::Q; ++q) f[q] = fo[q * N + idx] - L::w(q);
        if constexpr (TL::Q > 0) {
#pragma unroll
            for (int k = 0; k < TL::Q; ++k) g[k] = go[k * N + idx];
        }
        store_logical<L, TL, MASKED, PAT>(P, idx, o, m, f, g);
    } else {
        load_cell<L, TL, MASKED, PAT>(P, idx, o, m, f, g);
#pragma unroll
        for (int q = 0; q < L::Q; ++q) fo[q * N + idx] = f[q] + L::w(q);
        if constexpr (TL::Q > 0) {
            if (go) {
#pragma unroll
                for (int k = 0; k < TL::Q; ++k) go[k * N + idx] = g[k];
            }
        }
    }
}

// Diagnostics: per-block fp64 partial sums of
//   [0] sum (rho - 1), [1..3] sum j, [4..6] momentum exchange with solid cells,
//   [7..12] wall heat flux per Dirichlet face, [13] non-finite cells, [14] fluid cells,
//   [15..17] sum u_a T with u = (j + F/2)/rho (thermal lattices).
constexpr int DIAG_VALUES = 18;
constexpr int DIAG_N = 20;   // row stride of the partial sums
constexpr int DIAG_THREADS = 256;

constexpr int DIAG_CHUNK = 16;   // cells summed in fp32 before joining the fp64 totals

// The sums every fluid cell contributes (rho - 1, j, u T) run in fp32 over chunks of
// DIAG_CHUNK cells and join the fp64 totals once per chunk: GB300's fp64 rate is low enough
// that one fp64 add and conversion per value and cell would cost as much as the reads.
// The chunks' rounding (~1e-7 relative on sums of 16 deviation-sized values) stays far
// below the diagnostics' use.  Counts are integers; the rare wall and solid terms stay fp64.
template <class L, class TL, bool MASKED, int PAT>
__global__ void __launch_bounds__(DIAG_THREADS) diag_kernel(const Params P, double *partial)
{
    double acc[DIAG_VALUES];
#pragma unroll
    for (int i = 0; i < DIAG_VALUES; ++i) acc[i] = 0.0;
    float part[7] = {0, 0, 0, 0, 0, 0, 0};   // rho - 1, j, u T of the current chunk
    int in_chunk = 0, cells = 0, nonfinite = 0;
    auto flush = [&]() {
        acc[0] += part[0];
        acc[1] += part[1];
        acc[2] += part[2];
        acc[3] += part[3];
        acc[15] += part[4];
        acc[16] += part[5];
        acc[17] += part[6];
#pragma unroll
        for (int k = 0; k < 7; ++k) part[k] = 0.0f;
        in_chunk = 0;
    };
    const long long N = (long long)P.nx * P.ny * P.nz;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < N;
         i += (long long)gridDim.x * blockDim.x) {
        const int idx = (int)i;
        const int x = idx % P.nx;
        const int y = (idx / P.nx) % P.ny;
        const int z = idx / (P.nx * P.ny);
        uint32_t m = 0;
        if (MASKED) m = P.mask[idx];
        if ((m & SKIP_BITS) || (!MASKED && ghost_plane<L>(P, x, y, z))) continue;
        Offs o{};
        if (PAT != NATURAL) o = make_offs(x, y, z, P);
        float f[L::Q], g[TL::QA];
        load_cell<L, TL, MASKED, PAT>(P, idx, o, m, f, g);
        // per-cell sums in fp32 (GB300's fp64 rate is low), running totals in fp64
        float dr = 0.0f, jx = 0.0f, jy = 0.0f, jz = 0.0f, t = 0.0f;
#pragma unroll
        for (int q = 0; q < L::Q; ++q) {
            dr += f[q];
            if (L::cx(q)) jx += L::cx(q) * f[q];
            if (L::cy(q)) jy += L::cy(q) * f[q];
            if (L::cz(q)) jz += L::cz(q) * f[q];
        }
        part[0] += dr;
        part[1] += jx;
        part[2] += jy;
        part[3] += jz;
        if constexpr (TL::Q > 0) {
#pragma unroll
            for (int k = 0; k < TL::Q; ++k) t += g[k];
        }
        if (!isfinite(dr) || !isfinite(t)) ++nonfinite;
        ++cells;
        if constexpr (TL::Q > 0) {
            // convective transport, with the velocity of the macroscopic read-out
            float Fx, Fy, Fz, ux, uy, uz;
            force_velocity<true>(P.c, 1.0f + dr, t, jx, jy, jz, Fx, Fy, Fz, ux, uy, uz);
            part[4] += ux * t;
            part[5] += uy * t;
            part[6] += uz * t;
        }
        if (MASKED) {
            // links into solid cells: the bounced-back population of the last step is the
            // logical f_opp(q)(x) now; exchange 2 f+_q c_q
            const int c0[3] = {x, y, z};
            const int n[3] = {P.nx, P.ny, P.nz};
#pragma unroll
            for (int q = 1; q < L::Q; ++q) {
                if (!bit(m, q)) continue;
                const int c[3] = {L::cx(q), L::cy(q), L::cz(q)};
                bool face = false;
                for (int a = 0; a < 3; ++a) {
                    const int s = c0[a] + c[a];
                    if ((s < 0 && P.face_wall[2 * a]) || (s >= n[a] && P.face_wall[2 * a + 1]))
                        face = true;
                }
                if (face) continue;
                const double fp = (double)f[L::opp(q)] + (double)L::w(q);
                acc[4] += 2.0 * fp * c[0];
                acc[5] += 2.0 * fp * c[1];
                acc[6] += 2.0 * fp * c[2];
            }
        }
        if constexpr (TL::Q > 0) {
            const int c0[3] = {x, y, z};
            const int n[3] = {P.nx, P.ny, P.nz};
            for (int a = 0; a < L::DIM; ++a) {
                if (c0[a] == 0 && P.face_dir[2 * a]) acc[7 + 2 * a] += 2.0 * (P.T_wall[2 * a] - t);
                if (c0[a] == n[a] - 1 && P.face_dir[2 * a + 1])
                    acc[8 + 2 * a] += 2.0 * (P.T_wall[2 * a + 1] - t);
            }
        }
        if (++in_chunk == DIAG_CHUNK) flush();
    }
    flush();
    acc[13] = nonfinite;
    acc[14] = cells;
    // block reduction in a fixed order: warp shuffles, then warps in order
    __shared__ double sh[DIAG_THREADS / 32][DIAG_VALUES];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < DIAG_VALUES; ++i) {
        double v = acc[i];
        for (int s = 16; s > 0; s >>= 1) v += __shfl_down_sync(0xffffffffu, v, s);
        if (lane == 0) sh[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < DIAG_VALUES) {
        double v = 0.0;
        for (int w = 0; w < DIAG_THREADS / 32; ++w) v += sh[w][threadIdx.x];
        partial[blockIdx.x * DIAG_N + threadIdx.x] = v;
    }
}

// Sum the per-block partials in a fixed order into out[0..14].
static __global__ void __launch_bounds__(DIAG_THREADS) diag_finalize(const double *partial, int nblocks,
                                                               double *out)
{
    __shared__ double sh[DIAG_THREADS][DIAG_VALUES];
    double acc[DIAG_VALUES];
    for (int i = 0; i < DIAG_VALUES; ++i) acc[i] = 0.0;
    for (int b = threadIdx.x; b < nblocks; b += DIAG_THREADS)
        for (int i = 0; i < DIAG_VALUES; ++i) acc[i] += partial[b * DIAG_N + i];
    for (int i = 0; i < DIAG_VALUES; ++i) sh[threadIdx.x][i] = acc[i];
    __syncthreads();
    for (int s = DIAG_THREADS / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s)
            for (int i = 0; i < DIAG_VALUES; ++i) sh[threadIdx.x][i] += sh[threadIdx.x + s][i];
        __syncthreads();
    }
    if (threadIdx.x < DIAG_VALUES) out[threadIdx.x] = sh[0][threadIdx.x];
}

// ------------------------------------------------------------------ slab halos -------

// Halo exchange of a slab (HALO faces on the outer axis: z in 3-D, y in 2-D) or a block
// (HALO faces on any axes), with a ghost plane at each HALO face ("Multi-GPU thermal
// lattice Boltzmann simulations using OpenACC and MPI", Sec. 3: only the populations that
// cross a face are sent, as contiguous buffers).  Under the AA pattern only the odd step
// reads and writes across a face:
//   FILL  (before an odd step): the neighbour's boundary plane -> my ghost plane, the
//         populations pointing out through my face (they are what my boundary cells pull);
//   DRAIN (after it): my ghost plane -> the neighbour's boundary plane, the same populations
//         (what my boundary cells pushed into the ghost).
// A pack of side s / phase FILL reads my boundary plane at s with the populations pointing
// into my slab; unpack of side s / FILL writes my ghost plane at s with those pointing out;
// DRAIN swaps the planes' roles.  A plane spans the whole extent of the other axes, their
// ghost rows included: a block driver exchanges the axes one after another (the same order
// at FILL and at DRAIN), so that what crosses an edge or a corner travels through the ghost
// rows of the intermediate neighbours.  A DRAIN leaves slot (q, x) alone where
// the link of x towards the ghost (opposite q) is a wall link: x bounced that population
// back into the slot itself, and the ghost's copy was never written; and it leaves solid
// cells alone.  buf: [direction][plane cell], momentum then thermal; plane cells with the
// lower remaining axis fastest.
// Cell index of plane cell i (the lower remaining axis fastest) of the plane next to face
// `side` of AXIS: the ghost plane (ghost) or the first owned plane.
template <int AXIS>
LBM_HD int halo_plane_cell(const Params &P, int side, bool ghost, int i)
{
    const int n[3] = {P.nx, P.ny, P.nz};
    constexpr int u = AXIS == 0 ? 1 : 0, v = AXIS == 2 ? 1 : 2;
    int c3[3];
    c3[AXIS] = side ? n[AXIS] - 1 : 0;
    if (!ghost) c3[AXIS] += side ? -1 : 1;
    c3[u] = i % n[u];
    c3[v] = i / n[u];
    return c3[0] + P.nx * (c3[1] + P.ny * c3[2]);
}

template <class L, int AXIS>
LBM_HD constexpr int axis_c(int q)
{
    return AXIS == 0 ? L::cx(q) : AXIS == 1 ? L::cy(q) : L::cz(q);
}

// The slots of one cell that cross a face of AXIS in direction SIGN (c_AXIS = SIGN), held
// in registers: every load of a move is issued before its first store, since the source
// and the destination may be the same buffer and the compiler would otherwise keep each
// store behind the load before it.
template <class L, class TL>
struct HaloSlots {
    float f[L::Q], g[TL::QA];
};

template <class L, class TL, int AXIS, int SIGN>
LBM_HD void halo_load(const Params &S, int cell, HaloSlots<L, TL> &v)
{
#pragma unroll
    for (int q = 0; q < L::Q; ++q)
        if (axis_c<L, AXIS>(q) == SIGN) v.f[q] = S.f[(size_t)q * S.S + (unsigned)cell];
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int q = 0; q < TL::Q; ++q)   // thermal direction q is flow direction q
            if (axis_c<L, AXIS>(q) == SIGN) v.g[q] = S.g[(size_t)q * S.S + (unsigned)cell];
    }
}

// keep: the destination cell's mask on a DRAIN into an owned plane (else 0): a slot whose
// opposite link is a wall link keeps its value, and so does every slot of a solid cell.
template <class L, class TL, int AXIS, int SIGN>
LBM_HD void halo_store(const Params &D, int cell, uint32_t keep, const HaloSlots<L, TL> &v)
{
    if (keep & SOLID_BIT) return;
#pragma unroll
    for (int q = 0; q < L::Q; ++q)
        if (axis_c<L, AXIS>(q) == SIGN && !bit(keep, L::opp(q)))
            D.f[(size_t)q * D.S + (unsigned)cell] = v.f[q];
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int q = 0; q < TL::Q; ++q)
            if (axis_c<L, AXIS>(q) == SIGN && !bit(keep, L::opp(q)))
                D.g[(size_t)q * D.S + (unsigned)cell] = v.g[q];
    }
}

// The same slots to or from a contiguous buffer: [direction][plane cell], momentum then
// thermal, directions in index order.
template <class L, class TL, int AXIS, int SIGN>
LBM_HD void halo_to_buf(const HaloSlots<L, TL> &v, float *buf, int plane_cells, int i)
{
    int k = 0;
#pragma unroll
    for (int q = 0; q < L::Q; ++q)
        if (axis_c<L, AXIS>(q) == SIGN) buf[(size_t)(k++) * plane_cells + i] = v.f[q];
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int q = 0; q < TL::Q; ++q)
            if (axis_c<L, AXIS>(q) == SIGN) buf[(size_t)(k++) * plane_cells + i] = v.g[q];
    }
}

template <class L, class TL, int AXIS, int SIGN>
LBM_HD void halo_from_buf(const float *buf, int plane_cells, int i, HaloSlots<L, TL> &v)
{
    int k = 0;
#pragma unroll
    for (int q = 0; q < L::Q; ++q)
        if (axis_c<L, AXIS>(q) == SIGN) v.f[q] = buf[(size_t)(k++) * plane_cells + i];
    if constexpr (TL::Q > 0) {
#pragma unroll
        for (int q = 0; q < TL::Q; ++q)
            if (axis_c<L, AXIS>(q) == SIGN) v.g[q] = buf[(size_t)(k++) * plane_cells + i];
    }
}

template <int AXIS>
LBM_HD int halo_plane_cells(const Params &P)
{
    const int n[3] = {P.nx, P.ny, P.nz};
    return n[AXIS == 0 ? 1 : 0] * n[AXIS == 2 ? 1 : 2];
}

// Pack (unpack = 0) or unpack plane cell i of side `side` of AXIS in phase `phase`.
template <class L, class TL, int AXIS>
LBM_HD void halo_cell_axis(const Params &P, int side, int phase, int unpack, float *buf, int i)
{
    const int plane_cells = halo_plane_cells<AXIS>(P);
    // ghost plane of the side, or the owned plane next to it
    const bool ghost = (phase == 0) == (unpack != 0);
    const int idx = halo_plane_cell<AXIS>(P, side, ghost, i);
    // directions pointing out through the side (ghost plane) or into the block (owned plane)
    const int out_sign = side ? 1 : -1;
    const int sign = ghost ? out_sign : -out_sign;
    // DRAIN into my boundary plane: links that are bounced (or a solid cell) keep their own
    // value; a ghost cell on it (a block's edge) holds values in transit and takes them all
    const uint32_t keep = unpack && !ghost && P.mask ? P.mask[idx] : 0u;
    HaloSlots<L, TL> v;
    auto run = [&](auto sg) {
        constexpr int SG = decltype(sg)::value;
        if (!unpack) {
            halo_load<L, TL, AXIS, SG>(P, idx, v);
            halo_to_buf<L, TL, AXIS, SG>(v, buf, plane_cells, i);
        } else {
            halo_from_buf<L, TL, AXIS, SG>(buf, plane_cells, i, v);
            halo_store<L, TL, AXIS, SG>(P, idx, keep, v);
        }
    };
    if (sign > 0) run(std::integral_constant<int, 1>{});
    else run(std::integral_constant<int, -1>{});
}

template <class L, class TL>
LBM_HD void halo_cell(const Params &P, int axis, int side, int phase, int unpack, float *buf,
                      int i)
{
    if (axis == 0) halo_cell_axis<L, TL, 0>(P, side, phase, unpack, buf, i);
    else if (axis == 1) halo_cell_axis<L, TL, 1>(P, side, phase, unpack, buf, i);
    else halo_cell_axis<L, TL, 2>(P, side, phase, unpack, buf, i);
}

template <class L, class TL, int AXIS>
__global__ void halo_kernel(const Params P, int side, int phase, int unpack, float *buf)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < halo_plane_cells<AXIS>(P)) halo_cell_axis<L, TL, AXIS>(P, side, phase, unpack, buf, i);
}

// The exchange across one face without a buffer: block `lo`'s high face of AXIS meets block
// `hi`'s low face, both in memory this device can address.  Plane cell i, both ways:
// FILL: hi's first owned plane -> lo's ghost plane (slots with c_AXIS = +1), lo's first
//   owned plane -> hi's ghost plane (c_AXIS = -1);
// DRAIN: lo's ghost plane -> hi's first owned plane (c_AXIS = +1), hi's ghost plane -> lo's
//   first owned plane (c_AXIS = -1).
// It moves exactly what a pack on one side and an unpack on the other move.  Each move
// reads one plane of a block and writes another, so no thread reads a slot that another
// writes (lo may be hi: the two faces of a ring of one block, at least three planes thick).
template <class L, class TL, int AXIS>
LBM_HD void halo_swap_cell_axis(const Params &lo, const Params &hi, int phase, int i)
{
    const bool fill = phase == 0;
    // +1 direction: from hi (FILL: its owned plane) or lo (DRAIN: its ghost plane)
    const Params &s_up = fill ? hi : lo, &d_up = fill ? lo : hi;
    const int from_up = fill ? halo_plane_cell<AXIS>(hi, 0, false, i)
                             : halo_plane_cell<AXIS>(lo, 1, true, i);
    const int to_up = fill ? halo_plane_cell<AXIS>(lo, 1, true, i)
                           : halo_plane_cell<AXIS>(hi, 0, false, i);
    // -1 direction: from lo (FILL: its owned plane) or hi (DRAIN: its ghost plane)
    const Params &s_dn = fill ? lo : hi, &d_dn = fill ? hi : lo;
    const int from_dn = fill ? halo_plane_cell<AXIS>(lo, 1, false, i)
                             : halo_plane_cell<AXIS>(hi, 0, true, i);
    const int to_dn = fill ? halo_plane_cell<AXIS>(hi, 0, true, i)
                           : halo_plane_cell<AXIS>(lo, 1, false, i);
    const uint32_t keep_up = !fill && d_up.mask ? d_up.mask[to_up] : 0u;
    const uint32_t keep_dn = !fill && d_dn.mask ? d_dn.mask[to_dn] : 0u;
    HaloSlots<L, TL> up, dn;
    halo_load<L, TL, AXIS, 1>(s_up, from_up, up);
    halo_load<L, TL, AXIS, -1>(s_dn, from_dn, dn);
    halo_store<L, TL, AXIS, 1>(d_up, to_up, keep_up, up);
    halo_store<L, TL, AXIS, -1>(d_dn, to_dn, keep_dn, dn);
}

template <class L, class TL>
LBM_HD void halo_swap_cell(const Params &lo, const Params &hi, int axis, int phase, int i)
{
    if (axis == 0) halo_swap_cell_axis<L, TL, 0>(lo, hi, phase, i);
    else if (axis == 1) halo_swap_cell_axis<L, TL, 1>(lo, hi, phase, i);
    else halo_swap_cell_axis<L, TL, 2>(lo, hi, phase, i);
}

template <class L, class TL, int AXIS>
__global__ void halo_swap_kernel(const Params lo, const Params hi, int phase)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < halo_plane_cells<AXIS>(lo)) halo_swap_cell_axis<L, TL, AXIS>(lo, hi, phase, i);
}

}  // namespace lbm
