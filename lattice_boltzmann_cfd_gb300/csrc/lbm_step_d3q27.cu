// D3Q27 central-moment instantiations of the fused AA step kernel (no thermal lattice).
#include "lbm_internal.h"

namespace lbm {
namespace {

// The 32-bit-index forms without the immersed boundary fit the 27-population collision in
// 48 registers (5 blocks of 256 per SM) with at most a 4-byte spill; the extra warps hide
// memory latency in this issue-heavy kernel (periodic 512^3: 92.4 % -> 96.3 % of the copy
// bandwidth).  The 64-bit and immersed-boundary forms would spill there (up to 224 bytes)
// and keep the default bound.
template <bool M, bool O, bool N, bool I, bool F = false, bool B = false>
cudaError_t go(const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    if constexpr (N && !I)
        return launch_step_kernel(step_kernel_5<D3Q27, NoThermal, 2, M, O, N, I, F, B>, sh.grid,
                                  sh.block, s, chained, P);
    else
        return launch_step_kernel(step_kernel<D3Q27, NoThermal, 2, M, O, N, I, F, B>, sh.grid,
                                  sh.block, s, chained, P);
}

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t, bool);

// masked: 0 = no mask; 1 = mask, computed from the coordinates outside the solid cells'
// box and loaded inside it; 2 = the same with the box of the immersed-boundary samples'
// stencil cells included, and immersed-boundary forces
template <bool N>
cudaError_t dispatch_n(int masked, bool odd, bool box, const Params &P, const Shape &sh,
                       cudaStream_t s, bool chained)
{
    static const Fn table[3][2] = {{go<false, false, N, false>, go<false, true, N, false>},
                                   {go<true, false, N, false, true>, go<true, true, N, false, true>},
                                   {go<true, false, N, true, true>, go<true, true, N, true, true>}};
    // box launches (lbm_step_box) take no immersed boundary
    static const Fn boxed[2][2] = {
        {go<false, false, N, false, false, true>, go<false, true, N, false, false, true>},
        {go<true, false, N, false, true, true>, go<true, true, N, false, true, true>}};
    if (box) {
        if (masked > 1) return cudaErrorInvalidValue;
        return boxed[masked][odd ? 1 : 0](P, sh, s, chained);
    }
    return table[masked][odd ? 1 : 0](P, sh, s, chained);
}

}  // namespace

cudaError_t launch_step_d3q27(int masked, bool odd, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s, bool chained, bool box)
{
    return narrow ? dispatch_n<true>(masked, odd, box, P, sh, s, chained)
                  : dispatch_n<false>(masked, odd, box, P, sh, s, chained);
}

}  // namespace lbm
