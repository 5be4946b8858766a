"""Write ``cavity3d_512_walls.npz``: the fp64 oracle's state of the 512^3 side-heated
cavity (D3Q19 MRT + D3Q7 MRT, Ra = 1e7, Pr = 0.71, U_ff = 0.1, hot x = 0, cold x = L,
four adiabatic walls, buoyancy along +z; the cubic cell of "Multi-GPU thermal lattice
Boltzmann simulations using OpenACC and MPI", Sec. 4, at 512^3 instead of 385^3) after
200 and 201 steps, sampled next to the two Dirichlet walls.

Only the oracle runs here (with the seeded inputs of ``workloads.cavity3d``).  The whole
512^3 state in fp64 with the oracle's two buffers would need 56 GB, so each wall is run
on a window: x in [0, 209) for the hot wall and [303, 512) for the cold wall, with y and
z whole.  The oracle sets every population pulled from outside the window to NaN, and
information moves at most one cell per step, so after n <= 201 steps the 8 planes next to
the wall (x < 8, x >= 504) hold exactly the values of the whole-domain run.  The script
asserts that every stored value is finite.

Stored per wall ("hot", "cold") and step count n (200, 201), for 13 blocks of 4 x 4 cells
in (y, z) -- the four corners, the four edge centres, the face centre and four seeded
random blocks -- over the 8 planes next to the wall:
  ``{wall}_{n}_rho``  (13, 4, 4, 8), ``{wall}_{n}_u`` (13, 3, 4, 4, 8),
  ``{wall}_{n}_T``    (13, 4, 4, 8)      indexed [block, (component,) z, y, x-from-wall],
  ``{wall}_{n}_f``    (13, 19, 4, 4, 2), ``{wall}_{n}_g`` (13, 7, 4, 4, 2): the logical
                      populations of the 2 planes nearest the wall,
  ``{wall}_{n}_heat`` the wall's heat sum over its whole face, sum 2 (T_w - T_cell),
plus ``blocks`` (13, 2) = the (y0, z0) of each block and ``x_hot`` / ``x_cold`` = the x
indices of the 8 planes.

Run:  python tests/golden/make_cavity3d_512_walls.py   (about 90 minutes on 8 cores)
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from lattice_boltzmann_cfd_gb300 import workloads as W  # noqa: E402

N = 512
STEPS = (200, 201)
DEPTH = 8          # planes next to each wall whose values are exact after 201 steps
WIN = 201 + DEPTH  # window depth along x
B = 4              # block edge in y and z
OUT = os.path.join(HERE, "cavity3d_512_walls.npz")


def blocks():
    hi, mid = N - B, (N - B) // 2
    fixed = [(0, 0), (hi, 0), (0, hi), (hi, hi), (mid, 0), (mid, hi), (0, mid), (hi, mid),
             (mid, mid)]
    rng = np.random.default_rng(12)
    rand = [tuple(int(v) for v in rng.integers(0, N - B + 1, size=2)) for _ in range(4)]
    return np.array(fixed + rand, np.int64)


def main():
    w = W.cavity3d(n=N)
    blk = blocks()
    out = {"blocks": blk}
    face = {"hot": 0, "cold": 1}
    for wall, x0 in (("hot", 0), ("cold", N - WIN)):
        t0 = time.time()
        p = oracle.Problem(w, ((x0, 0, 0), (WIN, N, N)))
        f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
        xs = np.arange(DEPTH) if wall == "hot" else np.arange(WIN - 1, WIN - 1 - DEPTH, -1)
        out[f"x_{wall}"] = xs + x0
        done = 0
        for n in STEPS:
            oracle.run(p, f, g, n - done)
            done = n
            rho, u, T = oracle.macroscopic(p, f, g)
            d = oracle.diagnostics(p, f, g)
            heat = d["heat"][face[wall]]
            assert np.isfinite(heat)
            R = np.empty((len(blk), B, B, DEPTH))
            U = np.empty((len(blk), 3, B, B, DEPTH))
            TT = np.empty((len(blk), B, B, DEPTH))
            Fp = np.empty((len(blk), 19, B, B, 2))
            Gp = np.empty((len(blk), 7, B, B, 2))
            for i, (y0, z0) in enumerate(blk):
                sl = (slice(z0, z0 + B), slice(y0, y0 + B))
                R[i] = rho[sl][..., xs]
                U[i] = u[(slice(None),) + sl][..., xs]
                TT[i] = T[sl][..., xs]
                Fp[i] = f[(slice(None),) + sl][..., xs[:2]]
                Gp[i] = g[(slice(None),) + sl][..., xs[:2]]
            for k, v in (("rho", R), ("u", U), ("T", TT), ("f", Fp), ("g", Gp)):
                assert np.isfinite(v).all(), (wall, n, k)
                out[f"{wall}_{n}_{k}"] = v
            out[f"{wall}_{n}_heat"] = np.float64(heat)
            print(f"{wall} wall, {n} steps: heat {heat:.9e}, {time.time() - t0:.0f} s",
                  flush=True)
        del f, g, p
    np.savez_compressed(OUT, **out)
    print("wrote", OUT, os.path.getsize(OUT), "bytes")


if __name__ == "__main__":
    main()
