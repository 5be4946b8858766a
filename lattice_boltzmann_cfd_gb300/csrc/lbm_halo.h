// Batched face swaps between contexts on one device (lbm_halo_axis_swap_many): the compact
// per-context descriptor and the launcher.
#pragma once
#include "lbm_internal.h"

namespace lbm {

// What a face swap reads of one context, small enough for HALO_MAX_PAIRS pairs of them to
// travel as one kernel parameter (4 KB).
struct HaloSide {
    float *f, *g;
    const uint32_t *mask;
    size_t S;
    int nx, ny, nz;
    void from_params(const Params &P)
    {
        f = P.f;
        g = P.g;
        mask = P.mask;
        S = P.S;
        nx = P.nx;
        ny = P.ny;
        nz = P.nz;
    }
    LBM_HD void to_params(Params &P) const
    {
        P.f = f;
        P.g = g;
        P.mask = mask;
        P.S = S;
        P.nx = nx;
        P.ny = ny;
        P.nz = nz;
    }
};

constexpr int HALO_MAX_PAIRS = 32;

struct HaloPairs {
    HaloSide lo[HALO_MAX_PAIRS], hi[HALO_MAX_PAIRS];
    int n;
};
static_assert(sizeof(HaloPairs) <= 4000, "the pairs must fit the kernel parameter space");

// The face swaps of pairs.n pairs of one axis in one launch (halo_swap_many_kernel).
cudaError_t launch_halo_swap_many(int lattice, int thermal, const HaloPairs &pairs, int axis,
                                  int phase, cudaStream_t s);

}  // namespace lbm
