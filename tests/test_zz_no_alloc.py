"""The allocation-free reduction entry point, lbm_reduce_populations_static.

It serves callers that cannot call cudaMalloc (and so cannot hand the library a
workspace): it sums caller-held populations with its scratch in a static device array.
Its results must agree with the workspace-based lbm_diagnostics (mass, momentum) and with
the sum of the temperature field lbm_macroscopic writes, on two calls in a row (the
second call reuses the static scratch the first one left behind).

This file is collected last on purpose, so that a run that stops at the first failure
has run every other test first; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W

torch = pytest.importorskip("torch")


@pytest.mark.gpu
def test_static_reduction_matches_diagnostics_twice():
    from lattice_boltzmann_cfd_gb300 import Simulation, capi
    assert torch.cuda.is_available(), "CUDA device required"
    w = W.perturbed(W.cavity3d(shape=(70, 40, 36)), seed=5)
    solid = np.zeros(w.grid, np.uint8)
    solid[10:14, 12:18, 30:40] = 1
    w.solid = solid
    dev = torch.device("cuda")
    sim = Simulation(w)
    sim.init_equilibrium(torch.from_numpy(w.rho0).to(dev), torch.from_numpy(w.u0).to(dev),
                         torch.from_numpy(w.T_init).to(dev))
    out = torch.full((6,), float("nan"), dtype=torch.float64, device=dev)
    nx, ny, nz = w.shape
    for call, steps in enumerate((3, 4)):
        sim.step(steps)
        f, g = sim.populations()
        capi.lbm_reduce_populations_static(19, 7, nx, ny, nz, f, g, out)
        d = sim.diagnostics()
        T = sim.macroscopic()[2]
        r = out.cpu().numpy()
        # tolerances of the parity tests: mass 1e-6 relative, momentum 1e-4 relative
        assert np.isclose(r[0], d["mass"], rtol=1e-6, atol=0), (call, r[0], d["mass"])
        assert np.allclose(r[1:4], d["momentum"], rtol=1e-4, atol=1e-6 * d["mass"]), call
        T_sum = float(T.double().sum())
        assert np.isclose(r[4], T_sum, rtol=1e-4, atol=1e-3), (call, r[4], T_sum)
        assert r[5] == 0.0
    sim.close()
    lib = capi.load()
    big = 1 << 15
    st = lib.lbm_reduce_populations_static(19, 0, big, big, 1, out.data_ptr(), None,
                                           out.data_ptr(), None)
    assert st == capi.LBM_ERR_ARG
    assert "static scratch limit" in capi.lbm_last_error(None)
