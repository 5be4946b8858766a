"""Write ``periodic_512_window.npz``: the fp64 oracle's state of the periodic 512^3 D3Q19
MRT workload (``workloads.random_periodic(n=512, seed=2)``: rho = 1 + N(0, 1e-3), each
velocity component U(-0.02, 0.02), nu = 0.01, the other rates 1.2) after 200 and 201
steps, in an 8 x 8 x 8 block of cells.

Only the oracle runs here (with the seeded inputs of the workload).  The whole 512^3 state
in fp64 with the oracle's two buffers would need 41 GB, so the oracle runs on a window of
410^3 cells, the block plus 201 cells on every side.  It sets every population pulled from
outside the window to NaN, and information moves at most one cell per step, so after
n <= 201 steps the block holds exactly the values of the whole-domain run.  The script
asserts that every stored value is finite.

Stored for n in (200, 201):
  ``rho_{n}`` (8, 8, 8), ``u_{n}`` (3, 8, 8, 8), ``f_{n}`` (19, 8, 8, 8): fields and logical
  populations of the block, indexed [(component,) z, y, x],
plus ``origin`` = the (x, y, z) of the block's first cell.

Run:  python tests/golden/make_periodic_512_window.py   (about 40 minutes on 8 cores)
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

STEPS = (200, 201)
B = 8                       # block edge
MARGIN = 201                # cells a disturbance can travel in 201 steps
WIN = B + 2 * MARGIN        # window edge
W0 = 51                     # window origin on every axis: the block starts at 252
OUT = os.path.join(HERE, "periodic_512_window.npz")


def main():
    w = W.random_periodic(n=512, seed=2)
    t0 = time.time()
    p = oracle.Problem(w, ((W0, W0, W0), (WIN, WIN, WIN)))
    f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    blk = (slice(MARGIN, MARGIN + B),) * 3
    out = {"origin": np.array([W0 + MARGIN] * 3, np.int64)}
    done = 0
    for n in STEPS:
        oracle.run(p, f, g, n - done)
        done = n
        rho, u, _ = oracle.macroscopic(p, f, g)
        out[f"rho_{n}"] = np.array(rho[blk])
        out[f"u_{n}"] = np.array(u[(slice(None),) + blk])
        out[f"f_{n}"] = np.array(f[(slice(None),) + blk])
        for k in ("rho", "u", "f"):
            assert np.isfinite(out[f"{k}_{n}"]).all(), (n, k)
        print(f"{n} steps: rho mean {out[f'rho_{n}'].mean():.12f}, {time.time() - t0:.0f} s",
              flush=True)
    np.savez_compressed(OUT, **out)
    print(f"wrote {OUT} {os.path.getsize(OUT)} bytes")


if __name__ == "__main__":
    main()
