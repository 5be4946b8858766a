// D3Q19 (optionally + D3Q7) instantiations of the fused AA step kernel.
#include "lbm_internal.h"

namespace lbm {
namespace {

template <class TL, int C, bool M, bool O, bool N, bool I, bool F = false, bool B = false>
cudaError_t go(const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    return launch_step_kernel(step_kernel<D3Q19, TL, C, M, O, N, I, F, B>, sh.grid, sh.block, s,
                              chained, P);
}

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t, bool);

// masked: 0 = no mask; 1 = mask, computed from the coordinates outside the solid cells'
// box and loaded inside it; 2 = the same with the box of the immersed-boundary samples'
// stencil cells included, and immersed-boundary forces
template <class TL, bool N>
cudaError_t dispatch_n(int coll, int masked, bool odd, bool box, const Params &P,
                       const Shape &sh, cudaStream_t s, bool chained)
{
    static const Fn table[2][3][2] = {
        {{go<TL, 0, false, false, N, false>, go<TL, 0, false, true, N, false>},
         {go<TL, 0, true, false, N, false, true>, go<TL, 0, true, true, N, false, true>},
         {go<TL, 0, true, false, N, true, true>, go<TL, 0, true, true, N, true, true>}},
        {{go<TL, 1, false, false, N, false>, go<TL, 1, false, true, N, false>},
         {go<TL, 1, true, false, N, false, true>, go<TL, 1, true, true, N, false, true>},
         {go<TL, 1, true, false, N, true, true>, go<TL, 1, true, true, N, true, true>}}};
    // box launches (lbm_step_box) take no immersed boundary
    static const Fn boxed[2][2][2] = {
        {{go<TL, 0, false, false, N, false, false, true>, go<TL, 0, false, true, N, false, false, true>},
         {go<TL, 0, true, false, N, false, true, true>, go<TL, 0, true, true, N, false, true, true>}},
        {{go<TL, 1, false, false, N, false, false, true>, go<TL, 1, false, true, N, false, false, true>},
         {go<TL, 1, true, false, N, false, true, true>, go<TL, 1, true, true, N, false, true, true>}}};
    if (box) {
        if (masked > 1) return cudaErrorInvalidValue;
        return boxed[coll ? 1 : 0][masked][odd ? 1 : 0](P, sh, s, chained);
    }
    return table[coll ? 1 : 0][masked][odd ? 1 : 0](P, sh, s, chained);
}

template <class TL>
cudaError_t dispatch(int coll, int masked, bool odd, bool narrow, bool box, const Params &P,
                     const Shape &sh, cudaStream_t s, bool chained)
{
    return narrow ? dispatch_n<TL, true>(coll, masked, odd, box, P, sh, s, chained)
                  : dispatch_n<TL, false>(coll, masked, odd, box, P, sh, s, chained);
}

}  // namespace

cudaError_t launch_step_d3q19(int thermal, int coll, int masked, bool odd, bool narrow,
                              const Params &P, const Shape &sh, cudaStream_t s, bool chained,
                              bool box)
{
    if (thermal == 7) return dispatch<D3Q7>(coll, masked, odd, narrow, box, P, sh, s, chained);
    return dispatch<NoThermal>(coll, masked, odd, narrow, box, P, sh, s, chained);
}

}  // namespace lbm
