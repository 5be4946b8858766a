// D2Q9 (optionally + D2Q5) instantiations of the fused AA step kernel.
#include "lbm_internal.h"

namespace lbm {
namespace {

template <class TL, int C, bool M, bool O, bool N>
cudaError_t go(const Params &P, const Shape &sh, cudaStream_t s)
{
    step_kernel<D2Q9, TL, C, M, O, N><<<sh.grid, sh.block, 0, s>>>(P);
    return cudaGetLastError();
}

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t);

template <class TL, bool N>
cudaError_t dispatch_n(int coll, bool masked, bool odd, const Params &P, const Shape &sh,
                       cudaStream_t s)
{
    static const Fn table[2][2][2] = {
        {{go<TL, 0, false, false, N>, go<TL, 0, false, true, N>},
         {go<TL, 0, true, false, N>, go<TL, 0, true, true, N>}},
        {{go<TL, 1, false, false, N>, go<TL, 1, false, true, N>},
         {go<TL, 1, true, false, N>, go<TL, 1, true, true, N>}}};
    return table[coll ? 1 : 0][masked ? 1 : 0][odd ? 1 : 0](P, sh, s);
}

template <class TL>
cudaError_t dispatch(int coll, bool masked, bool odd, bool narrow, const Params &P,
                     const Shape &sh, cudaStream_t s)
{
    return narrow ? dispatch_n<TL, true>(coll, masked, odd, P, sh, s)
                  : dispatch_n<TL, false>(coll, masked, odd, P, sh, s);
}

}  // namespace

cudaError_t launch_step_d2q9(int thermal, int coll, bool masked, bool odd, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s)
{
    if (thermal == 5) return dispatch<D2Q5>(coll, masked, odd, narrow, P, sh, s);
    return dispatch<NoThermal>(coll, masked, odd, narrow, P, sh, s);
}

}  // namespace lbm
