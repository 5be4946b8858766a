"""The allocation-free reduction entry point, lbm_reduce_populations_static.

It serves callers that cannot call cudaMalloc (and so cannot hand the library a
workspace): it sums caller-held populations with its scratch in a static device array.
Its results must agree with the workspace-based lbm_diagnostics (mass, momentum) and with
the sum of the temperature field lbm_macroscopic writes, on two calls in a row (the
second call reuses the static scratch the first one left behind).  Every lattice
combination the entry point instantiates is run, with the result in device memory and in
page-locked host memory, and a planted NaN must be counted.

This file is collected last on purpose, so that a run that stops at the first failure
has run every other test first; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W

torch = pytest.importorskip("torch")


def _d3q19_d3q7():
    w = W.perturbed(W.cavity3d(shape=(70, 40, 36)), seed=5)
    solid = np.zeros(w.grid, np.uint8)
    solid[10:14, 12:18, 30:40] = 1
    w.solid = solid
    return w


CASES = {
    "d3q19_d3q7": _d3q19_d3q7,
    "d3q19": lambda: W.random_periodic(shape=(70, 33, 21), seed=6),
    "d2q9_d2q5": lambda: W.perturbed(W.cavity2d(shape=(300, 170, 1)), seed=7),
    "d2q9": lambda: W.random_periodic(shape=(300, 170, 1), seed=8, lattice=9),
    "d3q27": lambda: W.random_periodic(shape=(66, 30, 20), seed=9, lattice=27),
}


@pytest.mark.gpu
@pytest.mark.parametrize("host_out", [False, True], ids=["device_out", "pinned_out"])
@pytest.mark.parametrize("name", list(CASES))
def test_static_reduction_matches_diagnostics_twice(name, host_out):
    from lattice_boltzmann_cfd_gb300 import Simulation, capi
    assert torch.cuda.is_available(), "CUDA device required"
    w = CASES[name]()
    dev = torch.device("cuda")
    sim = Simulation(w)
    T0 = None if not w.thermal else torch.from_numpy(w.T_init).to(dev)
    sim.init_equilibrium(torch.from_numpy(w.rho0).to(dev), torch.from_numpy(w.u0).to(dev), T0)
    if host_out:
        out = torch.full((6,), float("nan"), dtype=torch.float64).pin_memory()
    else:
        out = torch.full((6,), float("nan"), dtype=torch.float64, device=dev)
    nx, ny, nz = w.shape
    for call, steps in enumerate((3, 4)):
        sim.step(steps)
        f, g = sim.populations()
        capi.lbm_reduce_populations_static(w.lattice, w.thermal, nx, ny, nz, f,
                                           g if w.thermal else None, out)
        torch.cuda.synchronize()
        d = sim.diagnostics()
        r = out.cpu().numpy().copy()
        # tolerances of the parity tests: mass 1e-6 relative, momentum 1e-4 relative
        assert np.isclose(r[0], d["mass"], rtol=1e-6, atol=0), (call, r[0], d["mass"])
        assert np.allclose(r[1:4], d["momentum"], rtol=1e-4, atol=1e-6 * d["mass"]), call
        if w.thermal:
            T_sum = float(sim.macroscopic()[2].double().sum())
            assert np.isclose(r[4], T_sum, rtol=1e-4, atol=1e-3), (call, r[4], T_sum)
        else:
            assert r[4] == 0.0
        assert r[5] == 0.0
    # a NaN in one population of one cell is counted once
    f, g = sim.populations()
    f.view(w.lattice, -1)[w.lattice - 1, 12345 % w.cells] = float("nan")
    capi.lbm_reduce_populations_static(w.lattice, w.thermal, nx, ny, nz, f,
                                       g if w.thermal else None, out)
    torch.cuda.synchronize()
    assert out.cpu().numpy()[5] == 1.0
    sim.close()


@pytest.mark.gpu
def test_static_reduction_rejects_bad_sizes():
    from lattice_boltzmann_cfd_gb300 import capi
    assert torch.cuda.is_available(), "CUDA device required"
    lib = capi.load()
    out = torch.zeros(6, dtype=torch.float64, device="cuda")
    p = out.data_ptr()
    big = 1 << 15
    # too many cells; and dimensions whose product overflows 64 bits
    for dims in ((big, big, 1), (2 ** 31 - 1, 2 ** 31 - 1, 2 ** 31 - 1), (1 << 29, 1, 1)):
        st = lib.lbm_reduce_populations_static(19, 0, *dims, p, None, p, None)
        assert st == capi.LBM_ERR_ARG, dims
        assert "static scratch limit" in capi.lbm_last_error(None)
    st = lib.lbm_reduce_populations_static(9, 0, 16, 16, 2, p, None, p, None)
    assert st == capi.LBM_ERR_ARG
    assert "nz == 1" in capi.lbm_last_error(None)
