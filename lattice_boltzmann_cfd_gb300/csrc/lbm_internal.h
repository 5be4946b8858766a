// Host-side launch interface between the C ABI (lbm_capi.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>

#include <utility>

#include "lbm_kernels.cuh"

namespace lbm {

// Launch a kernel that starts with wait_prerequisites().  chained: with programmatic stream
// serialization, so that it may be scheduled before the previous kernel in the stream
// completes (its blocks fill the SMs that the previous kernel's last wave leaves idle);
// otherwise an ordinary launch.
template <class... K, class... A>
cudaError_t launch_step_kernel(void (*kernel)(K...), dim3 grid, dim3 block, cudaStream_t s,
                               bool chained, A &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Whether the step kernels of a grid of `blocks` blocks are launched chained: only grids of
// at least two waves (16 resident blocks of 64 threads per SM).  Chaining gained 2-4 % on
// 128^3 grids (14 waves) and nothing at 512^3; on the 32^3 grid (512 blocks, part of one
// wave) it cost 8 %, with several launched grids resident and waiting at once.
inline bool chain_steps(long long blocks, int sms) { return blocks >= 2LL * 16 * sms; }

struct Shape {
    dim3 grid, block;
};

// One thread per cell, blocks of `threads` along x (rows of a block stacked in y when a
// row is shorter than the block).
// Blocks of 64 threads along x (rows of 32 stacked along y when nx <= 32).  Measured
// against 128- and 256-thread rows: the same on periodic 512^3, 1.7-4.6 % faster on the
// walled cavities (fewer blocks carry a divergent wall warp) and 6-9 % faster on 128^3
// grids (finer granularity at the end of a launch).
inline Shape cell_shape(int nx, int ny, int nz, int threads = 64)
{
    int bx = ((nx + 31) / 32) * 32;
    if (bx > threads) bx = threads;
    int by = threads / bx;
    if (by < 1) by = 1;
    Shape s;
    s.block = dim3(bx, by, 1);
    s.grid = dim3((nx + bx - 1) / bx, (ny + by - 1) / by, nz);
    return s;
}

// The AA step kernels' launch over the box of cells [lo, hi) (per axis x, y, z; in 2-D
// lo[2] = 0, hi[2] = 1).  linear (Params::linear): rows that are not a multiple of 32
// cells; it applies to boxes of whole outer-axis planes only (whole x, and whole y in 3-D):
// 64-thread blocks over the cells in storage order, along each z plane with one grid row
// per plane in 3-D, along the rows as one run in 2-D.  Otherwise cell_shape's blocks over
// the box.  *linear_out: whether the launch is linear.
inline Shape step_shape(int nx, int ny, int nz, int dim, const int lo[3], const int hi[3],
                        bool linear, bool *linear_out = nullptr)
{
    Shape s;
    const bool whole = lo[0] == 0 && hi[0] == nx && (dim == 2 || (lo[1] == 0 && hi[1] == ny));
    linear = linear && whole;
    if (linear_out) *linear_out = linear;
    if (linear) {
        s.block = dim3(64, 1, 1);
        if (dim == 3)
            s.grid = dim3((unsigned)(((long long)nx * ny + 63) / 64), (unsigned)(hi[2] - lo[2]), 1);
        else
            s.grid = dim3((unsigned)(((long long)nx * (hi[1] - lo[1]) + 63) / 64), 1, 1);
        return s;
    }
    s = cell_shape(hi[0] - lo[0], hi[1] - lo[1], dim == 3 ? hi[2] - lo[2] : 1);
    (void)nz;
    return s;
}

constexpr int DIAG_BLOCKS = 2048;   // capacity of the partial-sum rows (one resident wave at most)

// Each returns the launch error (cudaGetLastError) of what it enqueued.
// narrow: every population index fits in 32 bits (see slot()).  masked: 0 = no link
// mask, 1 = link mask, 2 = link mask and immersed-boundary forces.  The AA step kernels of
// forms 1 and 2 compute the mask from the coordinates outside the box of the solid cells
// (form 2: and of the samples' stencil cells) and load it inside (boxed_mask); the
// two-buffer kernels load it.
// chained: see launch_step_kernel.
// box: the launch covers the box [P.run_lo, P.run_hi) (lbm_step_box; masked 0 or 1 only),
// otherwise the whole grid.
cudaError_t launch_step_d3q19(int thermal, int coll, int masked, bool odd, bool narrow,
                              const Params &P, const Shape &sh, cudaStream_t s, bool chained,
                              bool box = false);
cudaError_t launch_step_d2q9(int thermal, int coll, int masked, bool odd, bool narrow,
                             const Params &P, const Shape &sh, cudaStream_t s, bool chained,
                             bool box = false);
// D3Q27, central moments, AA only; masked as above.
cudaError_t launch_step_d3q27(int masked, bool odd, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s, bool chained, bool box = false);
// Two-buffer modes: one PULL step, or one SPLIT step (collide + stream), from P.f/P.g
// into P.fo/P.go.
cudaError_t launch_pull_d3q19(int thermal, int coll, int masked, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s, bool chained);
cudaError_t launch_pull_d2q9(int thermal, int coll, int masked, bool narrow, const Params &P,
                             const Shape &sh, cudaStream_t s, bool chained);
cudaError_t launch_split_d3q19(int thermal, int coll, int masked, bool narrow, const Params &P,
                               const Shape &sh, cudaStream_t s, bool chained);
cudaError_t launch_split_d2q9(int thermal, int coll, int masked, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s, bool chained);
// pat: read pattern of the logical state (NATURAL, AA_ODD or PULL).
cudaError_t launch_init(int lattice, int thermal, int pat, const Params &P, const float *rho,
                        const float *u, const float *T, cudaStream_t s);
cudaError_t launch_mask(int lattice, int thermal, const Params &P, const uint8_t *solid,
                        uint32_t *mask, cudaStream_t s);
cudaError_t launch_macro(int lattice, int thermal, bool masked, int pat, const Params &P,
                         float *rho, float *u, float *T, cudaStream_t s);
cudaError_t launch_pop(int lattice, int thermal, bool masked, int pat, bool set,
                       const Params &P, float *f, float *g, cudaStream_t s);
// Immersed boundary: penalty + spreading for every sample (read pattern pat), and the
// IB_BIT marking of the samples' stencil cells.
cudaError_t launch_ib(int lattice, int thermal, int pat, const Params &P, cudaStream_t s,
                      bool chained);
// set: IB_BIT on the stencil cells of P's samples; otherwise cleared there.
cudaError_t launch_ib_mark(int lattice, const Params &P, uint32_t *mask, bool set,
                           cudaStream_t s);
// Device ordering of n caller samples (device addresses; ub, w may be null) into P's sample
// planes by l-block and Morton code (lbm_ib_order.cu); scratch: ib_order_scratch_bytes(cap)
// bytes, 256-byte aligned.  The number of dropped samples lands in ib_dropped_counter.
// Scratch of the device ordering: keys[2][cap] (64-bit), indices[2][cap], digit counts
// [256][tiles], the order of the last sort (perm[cap]: slot i holds caller sample perm[i]),
// and the dropped-sample count.
constexpr int IB_SORT_TILE = 2048;   // keys per block of the multi-block sort
inline size_t ib_sort_tiles(int cap) { return ((size_t)cap + IB_SORT_TILE - 1) / IB_SORT_TILE; }
inline size_t ib_order_scratch_bytes(int cap)
{
    return 2 * (size_t)cap * 8 + 3 * (size_t)cap * 4 + 256 * ib_sort_tiles(cap) * 4 + 256;
}
inline int *ib_order_perm(const Params &P, void *scratch)
{
    const size_t cap = (size_t)P.ib_cap;
    return reinterpret_cast<int *>(static_cast<char *>(scratch) + 2 * cap * 8 + 2 * cap * 4 +
                                   256 * ib_sort_tiles(P.ib_cap) * 4);
}
inline unsigned *ib_dropped_counter(const Params &P, void *scratch)
{
    return reinterpret_cast<unsigned *>(ib_order_perm(P, scratch) + P.ib_cap);
}
// reorder: sort the samples (and keep the order in perm); otherwise place them in the order
// of the last sort (perm), which must have had the same n.
cudaError_t launch_ib_order(int lattice, const Params &P, int n, int l, const float *xyz,
                            const float *ub, const float *w, void *scratch, bool reorder,
                            cudaStream_t s);
// Halo pack (unpack = 0) or unpack (unpack = 1) of one side of one axis, one phase.
cudaError_t launch_halo(int lattice, int thermal, const Params &P, int axis, int side,
                        int phase, int unpack, float *buf, cudaStream_t s);
// The buffer-free exchange of lo's high face with hi's low face on `axis` (halo_swap_kernel).
cudaError_t launch_halo_swap(int lattice, int thermal, const Params &lo, const Params &hi,
                             int axis, int phase, cudaStream_t s);
cudaError_t launch_diag(int lattice, int thermal, bool masked, int pat, const Params &P,
                        double *partial, double *out, cudaStream_t s);

}  // namespace lbm

// Record the error text returned by lbm_last_error(NULL) on this thread.
void lbm_internal_set_error(const char *msg);
