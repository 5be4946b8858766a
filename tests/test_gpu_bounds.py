"""Bounds of the CUDA path's accesses, on the GPU, in the launch geometry the library uses.

The library carves its state out of the caller's workspace: Q planes of S fp32 slots for f
(S = the cell count rounded up to 64), then the thermal planes, each region aligned to 256
bytes.  The slots [N, S) of every plane, the alignment gaps and anything past the end of
the workspace belong to no cell.  These tests fill them with a NaN bit pattern that no
kernel computes, run every kind of launch (both AA forms, captured graphs, box launches
with the linear and the row mapping, halo packs, unpacks and swaps, read-outs), and check
that every sentinel is intact: a write outside the cells would overwrite one, and a read
of one would turn a result into NaN (the tests check the state stays finite).  This is
the device-side counterpart of the host emulation's NaN guards.
"""
import dataclasses

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import capi
from lattice_boltzmann_cfd_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SENTINEL = 0x7FBADBAD      # a quiet NaN with a payload no arithmetic produces
EXTRA = 1 << 16            # bytes of workspace past the library's end


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    capi.load()


def _align(v):
    return (v + 255) // 256 * 256


def _guarded(w, monkeypatch, **kw):
    """A Simulation of ``w`` whose workspace has EXTRA bytes past the end, and the int32
    index ranges of its workspace that belong to no cell."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    probe = Simulation(w, **kw)
    nbytes = probe.nbytes
    probe.close()
    real = capi.lbm_workspace_bytes
    monkeypatch.setattr(capi, "lbm_workspace_bytes", lambda cfg: real(cfg) + EXTRA)
    sim = Simulation(w, **kw)
    monkeypatch.setattr(capi, "lbm_workspace_bytes", real)
    N = w.cells
    S = (N + 63) // 64 * 64
    Q, QT = w.lattice, w.thermal
    regions = []
    for q in range(Q):
        regions.append((q * S + N, (q + 1) * S))
    off_g = _align(Q * S * 4) // 4
    regions.append((Q * S, off_g))                       # gap after the f planes
    for k in range(QT):
        regions.append((off_g + k * S + N, off_g + (k + 1) * S))
    if QT:
        end_g = off_g + QT * S
        regions.append((end_g, _align(end_g * 4) // 4))  # gap after the g planes
    regions.append((nbytes // 4, (nbytes + EXTRA) // 4))  # past the library's end
    return sim, [(a, b) for a, b in regions if b > a]


def _arm(sim, regions):
    ws = sim.workspace.view(torch.int32)
    for a, b in regions:
        ws[a:b] = SENTINEL


def _intact(sim, regions):
    torch.cuda.synchronize()
    ws = sim.workspace.view(torch.int32)
    bad = sum(int((ws[a:b] != SENTINEL).sum()) for a, b in regions)
    return bad


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


CASES = [
    W.perturbed(W.cavity3d(shape=(70, 41, 37)), seed=111),            # walls, D3Q7, FACES
    W.random_periodic(shape=(66, 10, 9), seed=112),                    # linear launch
    dataclasses.replace(W.perturbed(W.cavity2d(shape=(300, 181, 1)), seed=113), gbeta=0.01),
    W.random_periodic(shape=(40, 12, 11), seed=114, lattice=27),
    W.perturbed(W.channel_sphere(shape=(90, 30, 27), center=(30, 15, 13), radius=5), seed=115),
    W.random_periodic(shape=(128, 64, 33), seed=116),                  # graph replay, N % 64 = 0
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_steps_stay_inside_the_cells(monkeypatch, w):
    """lbm_step (both forms; grids of at most 4 M cells replay captured graphs), box launches
    over a random partition, the read-outs and the population round trip write nothing
    outside the cells and read nothing there."""
    sim, regions = _guarded(w, monkeypatch)
    sim.init_equilibrium(_dev(w.rho0), _dev(w.u0), _dev(w.T_init))
    # the check sees a planted stray write (the last guarded word of each region)
    ws = sim.workspace.view(torch.int32)
    _arm(sim, regions)
    for a, b in regions:
        ws[b - 1] = 0
    assert _intact(sim, regions) == len(regions)
    _arm(sim, regions)
    sim.step(3)
    sim.step(70)                       # at least one 64-step graph where graphs apply
    ext = list(w.shape)
    rng = np.random.default_rng(7)
    for _ in range(2):                 # one even and one odd step through box launches
        cuts = []
        for a in range(3):
            k = min(2, ext[a] - 1)
            c = sorted(rng.choice(np.arange(1, ext[a]), size=k, replace=False)) if k else []
            e = [0] + [int(v) for v in c] + [ext[a]]
            cuts.append(list(zip(e[:-1], e[1:])))
        for x in cuts[0]:
            for y in cuts[1]:
                for z in cuts[2]:
                    sim.step_box((x[0], y[0], z[0]), (x[1], y[1], z[1]))
    n_outer = ext[w.dim - 1]
    sim.step_planes(0, n_outer // 2)   # whole planes: the linear mapping where it applies
    sim.step_planes(n_outer // 2, n_outer)
    rho, u, T = sim.macroscopic()
    f, g = sim.populations()
    sim.set_populations(f, g)
    d = sim.diagnostics()
    assert d["finite"]
    assert torch.isfinite(f).all() and torch.isfinite(rho).all()
    assert _intact(sim, regions) == 0
    sim.close()


def test_immersed_boundary_stays_inside_the_cells(monkeypatch):
    """The immersed-boundary kernels (interpolation, spreading with atomics, the sample
    ordering on the device) write nothing outside the cells' population planes."""
    w = W.channel_ib_sphere(shape=(40, 30, 26), center=(15.3, 14.7, 12.2), radius=5.1,
                            gx=1e-4, samples_per_area=2.0)
    edit = lambda cfg: setattr(cfg, "ib_max_samples", 4 * len(w.ib_x))
    sim, regions = _guarded(w, monkeypatch, edit=edit)
    sim.init_equilibrium(_dev(w.rho0), _dev(w.u0), _dev(w.T_init))
    _arm(sim, regions)
    sim.set_ib_samples(w.ib_x, w.ib_ub, w.ib_w)
    sim.step(9)
    x = torch.from_numpy(np.ascontiguousarray(w.ib_x, np.float32)).cuda()
    for k in range(4):
        sim.set_ib_samples_device(x + 0.1 * k, reorder=(k % 2 == 0))
        sim.step(1)
    assert sim.diagnostics()["finite"]
    assert _intact(sim, regions) == 0
    sim.close()


@pytest.mark.parametrize("nb", [(1, 1, 3), (2, 2, 1), (1, 2, 2)])
def test_halo_exchanges_stay_inside_the_cells(monkeypatch, nb):
    """Packs, unpacks and swaps of every axis (slabs and blocks, FILL and DRAIN) write
    nothing outside the cells of either context."""
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    w = W.perturbed(W.cavity3d(shape=(37, 29, 23)), seed=117)
    guards = {}
    real_init = Simulation.__init__

    def init(self, lw, *a, **kw):
        real = capi.lbm_workspace_bytes
        capi.lbm_workspace_bytes = lambda cfg: real(cfg) + EXTRA
        try:
            real_init(self, lw, *a, **kw)
        finally:
            capi.lbm_workspace_bytes = real
        N, Q, QT = lw.cells, lw.lattice, lw.thermal
        S = (N + 63) // 64 * 64
        off_g = _align(Q * S * 4) // 4
        regs = [(q * S + N, (q + 1) * S) for q in range(Q)] + [(Q * S, off_g)]
        regs += [(off_g + k * S + N, off_g + (k + 1) * S) for k in range(QT)]
        regs.append(((self.nbytes - EXTRA) // 4, self.nbytes // 4))
        guards[id(self)] = (self, [(a, b) for a, b in regs if b > a])

    monkeypatch.setattr(Simulation, "__init__", init)
    for exchange in ("swap", "buffers"):
        dom = BlockDomain(w, nb, exchange=exchange)
        dom.init_equilibrium()
        for sim, regs in guards.values():
            _arm(sim, regs)
        dom.step(5)
        f, _ = dom.populations()
        assert torch.isfinite(f).all()
        for sim, regs in guards.values():
            assert _intact(sim, regs) == 0, exchange
        dom.close()
        guards.clear()
