"""Choice of the immersed-boundary sample block edge by measurement.

"GPU Optimization for High-Quality Kinetic Fluid Simulation" (Sec. 4, Eq. 11) picks the block
edge l that the solid samples are grouped by as the one minimising the average cost of a step
over an interval of steps, enumerating l in {2, ..., L_m}, L_m the smallest edge of the
solid's bounding box.  (Its second parameter, the CSoA granularity alpha, belongs to a data
layout this library does not use.)  Here the cost is measured directly: for each candidate,
the same problem is set up with that edge, stepped, and timed with CUDA events.
"""
from __future__ import annotations

import numpy as np

from .solver import Simulation


def default_candidates(w, cap: int = 32):
    """{2, ..., min(L_m, cap)}, L_m the smallest edge of the samples' bounding box."""
    x = np.asarray(w.ib_x, dtype=np.float64).reshape(-1, 3)[:, :w.dim]
    edge = int(np.floor((x.max(axis=0) - x.min(axis=0)).min())) + 1
    return list(range(2, max(2, min(edge, cap)) + 1))


def search_ib_block(w, candidates=None, steps: int = 20, warmup: int = 4, device=None):
    """Time ``steps`` steps of workload ``w`` (which must carry immersed-boundary samples)
    for each candidate block edge; returns (best edge, {edge: ms per step})."""
    import torch
    if getattr(w, "ib_x", None) is None or not len(w.ib_x):
        raise ValueError("the workload has no immersed-boundary samples")
    candidates = list(candidates) if candidates else default_candidates(w)
    times = {}
    for edge in candidates:
        sim = Simulation(w, device=device, edit=lambda c, e=edge: setattr(c, "ib_block", e))
        dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(sim.device)
        sim.init_equilibrium(dev(w.rho0), dev(w.u0), dev(w.T_init) if w.thermal else None)
        sim.step(warmup)
        torch.cuda.synchronize(sim.device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        sim.step(steps)
        b.record()
        torch.cuda.synchronize(sim.device)
        times[edge] = a.elapsed_time(b) / steps
        sim.close()
    best = min(times, key=times.get)
    return best, times
