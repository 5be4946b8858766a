// D2Q9 (optionally + D2Q5) instantiations of the fused AA step kernel.
#include "lbm_internal.h"

namespace lbm {
namespace {

template <class TL, int C, bool M, bool O, bool N, bool I, bool F = false>
cudaError_t go(const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    return launch_step_kernel(step_kernel<D2Q9, TL, C, M, O, N, I, F>, sh.grid, sh.block, s, chained,
                              P);
}

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t, bool);

// masked: 0 = no mask; 1 = mask, computed from the coordinates outside the solid cells'
// box and loaded inside it; 2 = the same with the box of the immersed-boundary samples'
// stencil cells included, and immersed-boundary forces
template <class TL, bool N>
cudaError_t dispatch_n(int coll, int masked, bool odd, const Params &P, const Shape &sh,
                       cudaStream_t s, bool chained)
{
    static const Fn table[2][3][2] = {
        {{go<TL, 0, false, false, N, false>, go<TL, 0, false, true, N, false>},
         {go<TL, 0, true, false, N, false, true>, go<TL, 0, true, true, N, false, true>},
         {go<TL, 0, true, false, N, true, true>, go<TL, 0, true, true, N, true, true>}},
        {{go<TL, 1, false, false, N, false>, go<TL, 1, false, true, N, false>},
         {go<TL, 1, true, false, N, false, true>, go<TL, 1, true, true, N, false, true>},
         {go<TL, 1, true, false, N, true, true>, go<TL, 1, true, true, N, true, true>}}};
    return table[coll ? 1 : 0][masked][odd ? 1 : 0](P, sh, s, chained);
}

template <class TL>
cudaError_t dispatch(int coll, int masked, bool odd, bool narrow, const Params &P,
                     const Shape &sh, cudaStream_t s, bool chained)
{
    return narrow ? dispatch_n<TL, true>(coll, masked, odd, P, sh, s, chained)
                  : dispatch_n<TL, false>(coll, masked, odd, P, sh, s, chained);
}

}  // namespace

cudaError_t launch_step_d2q9(int thermal, int coll, int masked, bool odd, bool narrow,
                              const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    if (thermal == 5) return dispatch<D2Q5>(coll, masked, odd, narrow, P, sh, s, chained);
    return dispatch<NoThermal>(coll, masked, odd, narrow, P, sh, s, chained);
}

}  // namespace lbm
