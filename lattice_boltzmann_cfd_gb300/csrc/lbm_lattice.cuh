// Lattice descriptors of the CUDA path: velocity sets, weights and opposites, as
// compile-time functions so that unrolled direction loops fold to constants.
//
// Orders: D3Q19 in d'Humieres' order (rest; +-x, +-y, +-z; xy, xz, yz edge links, each
// group (+,+), (-,+), (+,-), (-,-)); D2Q9 as the thermal multi-GPU LBM page's halo
// description implies (f2, f5, f6 cross the top face, f4, f7, f8 the bottom one);
// D3Q7 and D2Q5 share their axis directions' indices with D3Q19 and D2Q9.
#pragma once

#define LBM_HD __host__ __device__ __forceinline__

namespace lbm {

struct D3Q19 {
    static constexpr int Q = 19, DIM = 3;
    LBM_HD static constexpr int cx(int q) {
        constexpr int t[19] = {0, 1, -1, 0, 0, 0, 0, 1, -1, 1, -1, 1, -1, 1, -1, 0, 0, 0, 0};
        return t[q];
    }
    LBM_HD static constexpr int cy(int q) {
        constexpr int t[19] = {0, 0, 0, 1, -1, 0, 0, 1, 1, -1, -1, 0, 0, 0, 0, 1, -1, 1, -1};
        return t[q];
    }
    LBM_HD static constexpr int cz(int q) {
        constexpr int t[19] = {0, 0, 0, 0, 0, 1, -1, 0, 0, 0, 0, 1, 1, -1, -1, 1, 1, -1, -1};
        return t[q];
    }
    LBM_HD static constexpr int opp(int q) {
        constexpr int t[19] = {0, 2, 1, 4, 3, 6, 5, 10, 9, 8, 7, 14, 13, 12, 11, 18, 17, 16, 15};
        return t[q];
    }
    LBM_HD static constexpr float w(int q) {
        return q == 0 ? 1.0f / 3.0f : (q <= 6 ? 1.0f / 18.0f : 1.0f / 36.0f);
    }
};

struct D2Q9 {
    static constexpr int Q = 9, DIM = 2;
    LBM_HD static constexpr int cx(int q) {
        constexpr int t[9] = {0, 1, 0, -1, 0, 1, -1, -1, 1};
        return t[q];
    }
    LBM_HD static constexpr int cy(int q) {
        constexpr int t[9] = {0, 0, 1, 0, -1, 1, 1, -1, -1};
        return t[q];
    }
    LBM_HD static constexpr int cz(int) { return 0; }
    LBM_HD static constexpr int opp(int q) {
        constexpr int t[9] = {0, 3, 4, 1, 2, 7, 8, 5, 6};
        return t[q];
    }
    LBM_HD static constexpr float w(int q) {
        return q == 0 ? 4.0f / 9.0f : (q <= 4 ? 1.0f / 9.0f : 1.0f / 36.0f);
    }
};

// D3Q27 (every c in {-1, 0, 1}^3): D3Q19's order, then the corners (+,+,+), (-,+,+),
// (+,-,+), (-,-,+), (+,+,-), (-,+,-), (+,-,-), (-,-,-).  Weights are products of the D1Q3
// weights 2/3 (rest) and 1/6 (moving).
struct D3Q27 {
    static constexpr int Q = 27, DIM = 3;
    LBM_HD static constexpr int cx(int q) {
        constexpr int t[27] = {0, 1, -1, 0, 0, 0, 0, 1, -1, 1, -1, 1, -1, 1, -1, 0, 0, 0, 0,
                               1, -1, 1, -1, 1, -1, 1, -1};
        return t[q];
    }
    LBM_HD static constexpr int cy(int q) {
        constexpr int t[27] = {0, 0, 0, 1, -1, 0, 0, 1, 1, -1, -1, 0, 0, 0, 0, 1, -1, 1, -1,
                               1, 1, -1, -1, 1, 1, -1, -1};
        return t[q];
    }
    LBM_HD static constexpr int cz(int q) {
        constexpr int t[27] = {0, 0, 0, 0, 0, 1, -1, 0, 0, 0, 0, 1, 1, -1, -1, 1, 1, -1, -1,
                               1, 1, 1, 1, -1, -1, -1, -1};
        return t[q];
    }
    LBM_HD static constexpr int opp(int q) {
        constexpr int t[27] = {0, 2, 1, 4, 3, 6, 5, 10, 9, 8, 7, 14, 13, 12, 11, 18, 17, 16, 15,
                               26, 25, 24, 23, 22, 21, 20, 19};
        return t[q];
    }
    LBM_HD static constexpr float w(int q) {
        return q == 0 ? 8.0f / 27.0f
                      : (q <= 6 ? 2.0f / 27.0f : (q <= 18 ? 1.0f / 54.0f : 1.0f / 216.0f));
    }
};

// Thermal lattices: Q = 0 means "no thermal populations"; QA is the array size to use.
struct NoThermal {
    static constexpr int Q = 0, QA = 1;
};
struct D3Q7 {
    static constexpr int Q = 7, QA = 7;
};
struct D2Q5 {
    static constexpr int Q = 5, QA = 5;
};

// Face index (-x, +x, -y, +y, -z, +z = 0..5) a link of direction (cx, cy, cz) leaves
// through, for axis links.
LBM_HD constexpr int axis_face(int cx, int cy, int cz) {
    return cx > 0 ? 1 : cx < 0 ? 0 : cy > 0 ? 3 : cy < 0 ? 2 : cz > 0 ? 5 : 4;
}

// Per-cell link mask bits.
constexpr unsigned SOLID_BIT = 1u << 31;
constexpr unsigned IB_BIT = 1u << 30;   // the cell receives immersed-boundary force
constexpr unsigned GHOST_BIT = 1u << 29;  // halo plane of a slab (holds a neighbour's slots)
constexpr unsigned SKIP_BITS = SOLID_BIT | GHOST_BIT;   // cells that are never updated
constexpr int DIRICHLET_SHIFT = 19;   // bit 19 + k: thermal link k ends on a Dirichlet face

}  // namespace lbm
