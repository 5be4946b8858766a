// D2Q9 (optionally + D2Q5) instantiations of the two-buffer modes (PULL and SPLIT).
#include "lbm_internal.h"

namespace lbm {
namespace {

using Fn = cudaError_t (*)(const Params &, const Shape &, cudaStream_t, bool);

template <class TL, int C, bool M, bool N, bool I>
cudaError_t pull(const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    return launch_step_kernel(pull_kernel<D2Q9, TL, C, M, N, I>, sh.grid, sh.block, s, chained, P);
}

template <class TL, int C, bool M, bool N, bool I>
cudaError_t split(const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    cudaError_t e = launch_step_kernel(collide_kernel<D2Q9, TL, C, M, N, I>, sh.grid, sh.block, s,
                                       chained, P);
    if (e != cudaSuccess) return e;
    return launch_step_kernel(stream_kernel<D2Q9, TL, M, N>, sh.grid, sh.block, s, chained, P);
}

// masked: 0 = no mask, 1 = mask, 2 = mask and immersed-boundary forces
template <class TL, bool PULL_MODE>
cudaError_t dispatch(int coll, int masked, bool narrow, const Params &P, const Shape &sh,
                     cudaStream_t s, bool chained)
{
#define LBM_ENTRY(C, M, N, I) (PULL_MODE ? pull<TL, C, M, N, I> : split<TL, C, M, N, I>)
    static const Fn table[2][3][2] = {
        {{LBM_ENTRY(0, false, false, false), LBM_ENTRY(0, false, true, false)},
         {LBM_ENTRY(0, true, false, false), LBM_ENTRY(0, true, true, false)},
         {LBM_ENTRY(0, true, false, true), LBM_ENTRY(0, true, true, true)}},
        {{LBM_ENTRY(1, false, false, false), LBM_ENTRY(1, false, true, false)},
         {LBM_ENTRY(1, true, false, false), LBM_ENTRY(1, true, true, false)},
         {LBM_ENTRY(1, true, false, true), LBM_ENTRY(1, true, true, true)}}};
#undef LBM_ENTRY
    return table[coll ? 1 : 0][masked][narrow ? 1 : 0](P, sh, s, chained);
}

}  // namespace

cudaError_t launch_pull_d2q9(int thermal, int coll, int masked, bool narrow,
                             const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    if (thermal == 5) return dispatch<D2Q5, true>(coll, masked, narrow, P, sh, s, chained);
    return dispatch<NoThermal, true>(coll, masked, narrow, P, sh, s, chained);
}

cudaError_t launch_split_d2q9(int thermal, int coll, int masked, bool narrow,
                              const Params &P, const Shape &sh, cudaStream_t s, bool chained)
{
    if (thermal == 5) return dispatch<D2Q5, false>(coll, masked, narrow, P, sh, s, chained);
    return dispatch<NoThermal, false>(coll, masked, narrow, P, sh, s, chained);
}

}  // namespace lbm
