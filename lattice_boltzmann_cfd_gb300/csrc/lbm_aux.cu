// Launchers of the auxiliary kernels (initialisation, mask, read-out, diagnostics) for
// both lattices.
#include <type_traits>

#include "lbm_internal.h"
#include "lbm_halo.h"

namespace lbm {
namespace {

// Call fn(L{}, TL{}) with the momentum and thermal lattice types of a context.
template <class Fn>
cudaError_t by_lattice(int lattice, int thermal, Fn &&fn)
{
    if (lattice == 19) {
        if (thermal == 7) return fn(D3Q19{}, D3Q7{});
        return fn(D3Q19{}, NoThermal{});
    }
    if (lattice == 27) return fn(D3Q27{}, NoThermal{});
    if (thermal == 5) return fn(D2Q9{}, D2Q5{});
    return fn(D2Q9{}, NoThermal{});
}

Shape shape_of(const Params &P) { return cell_shape(P.nx, P.ny, P.nz); }

}  // namespace

namespace {
template <class L, class TL>
cudaError_t init_go(int pat, const Params &P, const float *rho, const float *u, const float *T,
                    cudaStream_t s)
{
    const Shape sh = shape_of(P);
    if (pat == PULL) init_kernel<L, TL, PULL><<<sh.grid, sh.block, 0, s>>>(P, rho, u, T);
    else init_kernel<L, TL, NATURAL><<<sh.grid, sh.block, 0, s>>>(P, rho, u, T);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_init(int lattice, int thermal, int pat, const Params &P, const float *rho,
                        const float *u, const float *T, cudaStream_t s)
{
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        return init_go<decltype(l), decltype(tl)>(pat, P, rho, u, T, s);
    });
}

cudaError_t launch_mask(int lattice, int thermal, const Params &P, const uint8_t *solid,
                        uint32_t *mask, cudaStream_t s)
{
    const Shape sh = shape_of(P);
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        mask_kernel<decltype(l), decltype(tl)><<<sh.grid, sh.block, 0, s>>>(P, solid, mask);
        return cudaGetLastError();
    });
}

cudaError_t launch_ib(int lattice, int thermal, int pat, const Params &P, cudaStream_t s,
                      bool chained)
{
    if (P.ib_n <= 0) return cudaSuccess;
    const int corners = lattice == 9 ? 4 : 8;
    const long long threads = (long long)P.ib_n * corners;
    const dim3 b(128), g((unsigned)((threads + 127) / 128));
    auto go = [&](auto l, auto tl) {
        using L = decltype(l);
        using TL = decltype(tl);
        if (pat == AA_ODD) return launch_step_kernel(ib_kernel<L, TL, AA_ODD>, g, b, s, chained, P);
        if (pat == PULL) return launch_step_kernel(ib_kernel<L, TL, PULL>, g, b, s, chained, P);
        return launch_step_kernel(ib_kernel<L, TL, NATURAL>, g, b, s, chained, P);
    };
    return by_lattice(lattice, thermal, go);
}

cudaError_t launch_ib_mark(int lattice, const Params &P, uint32_t *mask, bool set,
                           cudaStream_t s)
{
    int *box = const_cast<int *>(P.ib_box);
    if (set) {   // an empty box: every entry very negative
        cudaError_t e = cudaMemsetAsync(box, 0x80, 6 * sizeof(int), s);
        if (e != cudaSuccess) return e;
    }
    if (P.ib_n <= 0) return cudaSuccess;
    const dim3 b(128), g((P.ib_n + 127) / 128);
    auto go = [&](auto l) {
        using L = decltype(l);
        if (set) ib_mark_kernel<L, true><<<g, b, 0, s>>>(P, mask, box);
        else ib_mark_kernel<L, false><<<g, b, 0, s>>>(P, mask, box);
    };
    if (lattice == 19) go(D3Q19{});
    else if (lattice == 27) go(D3Q27{});
    else go(D2Q9{});
    return cudaGetLastError();
}

// Halo kernels move a plane of cells with a few slots each: small blocks spread a plane over
// more SMs, which keeps more loads in flight.
constexpr int HALO_THREADS = 128;

cudaError_t launch_halo(int lattice, int thermal, const Params &P, int axis, int side,
                        int phase, int unpack, float *buf, cudaStream_t s)
{
    const int n[3] = {P.nx, P.ny, P.nz};
    const int plane_cells = n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
    const dim3 b(HALO_THREADS), g((plane_cells + HALO_THREADS - 1) / HALO_THREADS);
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        using Lt = decltype(l);
        using Tt = decltype(tl);
        if (axis == 0) halo_kernel<Lt, Tt, 0><<<g, b, 0, s>>>(P, side, phase, unpack, buf);
        else if (axis == 1) halo_kernel<Lt, Tt, 1><<<g, b, 0, s>>>(P, side, phase, unpack, buf);
        else halo_kernel<Lt, Tt, 2><<<g, b, 0, s>>>(P, side, phase, unpack, buf);
        return cudaGetLastError();
    });
}

cudaError_t launch_halo_swap(int lattice, int thermal, const Params &lo, const Params &hi,
                             int axis, int phase, cudaStream_t s)
{
    const int n[3] = {lo.nx, lo.ny, lo.nz};
    const int plane_cells = n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
    const dim3 b(HALO_THREADS), g((plane_cells + HALO_THREADS - 1) / HALO_THREADS);
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        using Lt = decltype(l);
        using Tt = decltype(tl);
        if (axis == 0) halo_swap_kernel<Lt, Tt, 0><<<g, b, 0, s>>>(lo, hi, phase);
        else if (axis == 1) halo_swap_kernel<Lt, Tt, 1><<<g, b, 0, s>>>(lo, hi, phase);
        else halo_swap_kernel<Lt, Tt, 2><<<g, b, 0, s>>>(lo, hi, phase);
        return cudaGetLastError();
    });
}

namespace {

// Several face swaps of one axis in one launch: grid row p moves pair p.  The pairs of one
// axis touch disjoint slots (a block that is `hi` of one pair and `lo` of the next reads its
// first owned planes on both sides but writes other planes, or other slots of them), so the
// order of the swaps within an axis does not matter.
template <class L, class TL, int AXIS>
__global__ void halo_swap_many_kernel(const HaloPairs pairs, int phase)
{
    const int p = blockIdx.y;
    if (p >= pairs.n) return;
    Params lo{}, hi{};
    pairs.lo[p].to_params(lo);
    pairs.hi[p].to_params(hi);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < halo_plane_cells<AXIS>(lo)) halo_swap_cell_axis<L, TL, AXIS>(lo, hi, phase, i);
}

}  // namespace

cudaError_t launch_halo_swap_many(int lattice, int thermal, const HaloPairs &pairs, int axis,
                                  int phase, cudaStream_t s)
{
    int most = 0;
    for (int p = 0; p < pairs.n; ++p) {
        const int n[3] = {pairs.lo[p].nx, pairs.lo[p].ny, pairs.lo[p].nz};
        const int cells = n[axis == 0 ? 1 : 0] * n[axis == 2 ? 1 : 2];
        most = cells > most ? cells : most;
    }
    const dim3 b(HALO_THREADS), g((most + HALO_THREADS - 1) / HALO_THREADS, pairs.n);
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        using Lt = decltype(l);
        using Tt = decltype(tl);
        if (axis == 0) halo_swap_many_kernel<Lt, Tt, 0><<<g, b, 0, s>>>(pairs, phase);
        else if (axis == 1) halo_swap_many_kernel<Lt, Tt, 1><<<g, b, 0, s>>>(pairs, phase);
        else halo_swap_many_kernel<Lt, Tt, 2><<<g, b, 0, s>>>(pairs, phase);
        return cudaGetLastError();
    });
}

namespace {
// Call fn with compile-time (MASKED, PAT).
template <class Fn>
void with_pattern(bool masked, int pat, Fn &&fn)
{
    auto by_pat = [&](auto m) {
        if (pat == AA_ODD) fn(m, std::integral_constant<int, AA_ODD>{});
        else if (pat == PULL) fn(m, std::integral_constant<int, PULL>{});
        else fn(m, std::integral_constant<int, NATURAL>{});
    };
    if (masked) by_pat(std::true_type{});
    else by_pat(std::false_type{});
}

template <class L, class TL>
cudaError_t macro_go(bool masked, int pat, const Params &P, float *rho, float *u, float *T,
                     cudaStream_t s)
{
    const Shape sh = shape_of(P);
    with_pattern(masked, pat, [&](auto m, auto p) {
        macro_kernel<L, TL, decltype(m)::value, decltype(p)::value>
            <<<sh.grid, sh.block, 0, s>>>(P, rho, u, T);
    });
    return cudaGetLastError();
}

template <class L, class TL, bool SET>
cudaError_t pop_go(bool masked, int pat, const Params &P, float *f, float *g, cudaStream_t s)
{
    const Shape sh = shape_of(P);
    with_pattern(masked, pat, [&](auto m, auto p) {
        pop_kernel<L, TL, decltype(m)::value, decltype(p)::value, SET>
            <<<sh.grid, sh.block, 0, s>>>(P, f, g);
    });
    return cudaGetLastError();
}

// Blocks of a grid-stride kernel that make exactly one resident wave on this device (every
// block then does the same share of the work, and none waits for a second wave).
template <class K>
int one_wave(K kernel, int threads, int cap)
{
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        sms * per_sm < 1)
        return cap;
    return sms * per_sm < cap ? sms * per_sm : cap;
}

template <class L, class TL>
cudaError_t diag_go(bool masked, int pat, const Params &P, double *partial, double *out,
                    cudaStream_t s)
{
    int blocks = DIAG_BLOCKS;
    with_pattern(masked, pat, [&](auto m, auto p) {
        auto kernel = diag_kernel<L, TL, decltype(m)::value, decltype(p)::value>;
        blocks = one_wave(kernel, DIAG_THREADS, DIAG_BLOCKS);
        kernel<<<blocks, DIAG_THREADS, 0, s>>>(P, partial);
    });
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    diag_finalize<<<1, DIAG_THREADS, 0, s>>>(partial, blocks, out);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_macro(int lattice, int thermal, bool masked, int pat, const Params &P,
                         float *rho, float *u, float *T, cudaStream_t s)
{
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        return macro_go<decltype(l), decltype(tl)>(masked, pat, P, rho, u, T, s);
    });
}

cudaError_t launch_pop(int lattice, int thermal, bool masked, int pat, bool set,
                       const Params &P, float *f, float *g, cudaStream_t s)
{
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        using L = decltype(l);
        using TL = decltype(tl);
        return set ? pop_go<L, TL, true>(masked, pat, P, f, g, s)
                   : pop_go<L, TL, false>(masked, pat, P, f, g, s);
    });
}

cudaError_t launch_diag(int lattice, int thermal, bool masked, int pat, const Params &P,
                        double *partial, double *out, cudaStream_t s)
{
    return by_lattice(lattice, thermal, [&](auto l, auto tl) {
        return diag_go<decltype(l), decltype(tl)>(masked, pat, P, partial, out, s);
    });
}

}  // namespace lbm
