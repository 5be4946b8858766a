// D3Q27 central-moment instantiations of the fused AA step kernel (no thermal lattice, no
// immersed boundary).
#include "lbm_internal.h"

namespace lbm {
namespace {

template <bool M, bool O, bool N>
cudaError_t go(const Params &P, const Shape &sh, cudaStream_t s)
{
    step_kernel<D3Q27, NoThermal, 2, M, O, N, false><<<sh.grid, sh.block, 0, s>>>(P);
    return cudaGetLastError();
}

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t);

template <bool N>
cudaError_t dispatch_n(bool masked, bool odd, const Params &P, const Shape &sh,
                       cudaStream_t s)
{
    static const Fn table[2][2] = {{go<false, false, N>, go<false, true, N>},
                                   {go<true, false, N>, go<true, true, N>}};
    return table[masked ? 1 : 0][odd ? 1 : 0](P, sh, s);
}

}  // namespace

cudaError_t launch_step_d3q27(int masked, bool odd, bool narrow, const Params &P,
                              const Shape &sh, cudaStream_t s)
{
    if (masked > 1) return cudaErrorNotSupported;   // no immersed boundary on D3Q27
    return narrow ? dispatch_n<true>(masked != 0, odd, P, sh, s)
                  : dispatch_n<false>(masked != 0, odd, P, sh, s);
}

}  // namespace lbm
