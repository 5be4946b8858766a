"""Slab decomposition along the outer axis with the direction-selective halo exchange, on the
GPU through the C ABI: the slabs together hold bit for bit the state of one domain run with
the same kernels, at both AA parities, and their summed diagnostics agree with it.

In these cases every slab runs the same kernel family as the undivided domain (masked where
the domain has walls or solids on its other axes, unmasked where it is periodic and
all-fluid), so the comparison is between identical per-cell arithmetic and any difference
is an exchange error.  Every slab run is also compared element by element with the fp64
oracle run on the undivided domain.  A domain whose only walls close the outer axis mixes
the two families (the end slabs are masked, the inner ones are not); it is compared with
the undivided domain within fp32 rounding."""
import dataclasses

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import capi
from lattice_boltzmann_cfd_gb300 import workloads as W
from parity_util import (TOL_FIELDS, compare_fields, oracle_states, outer_walls_case,
                         slab_cases)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    capi.load()


def _single(w, steps):
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    sim = Simulation(w)
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sim.init_equilibrium(dev(w.rho0), dev(w.u0), dev(w.T_init))
    sim.step(steps)
    f, g = sim.populations()
    out = (f.cpu().numpy(), None if g is None else g.cpu().numpy(), sim.diagnostics())
    sim.close()
    return out


def _slabs(w, steps, nslabs, chunks=None, fields=False, exchange="auto"):
    """(f, g, diagnostics) of the slab run, plus its (rho, u, T) when ``fields``."""
    from lattice_boltzmann_cfd_gb300.slabs import SlabDomain
    dom = SlabDomain(w, nslabs, exchange=exchange)
    dom.init_equilibrium()
    for c in chunks or [steps]:
        dom.step(c)
    f, g = dom.populations()
    out = (f.cpu().numpy(), None if g is None else g.cpu().numpy(), dom.diagnostics())
    if fields:
        rho, u, T = dom.macroscopic()
        out += ({"rho": rho.cpu().numpy(), "u": u.cpu().numpy(),
                 "T": None if T is None else T.cpu().numpy(), "f": out[0], "g": out[1]},)
    dom.close()
    return out


def _large_cases():
    """Grids spanning several thread blocks along x with ragged tails and uneven slabs."""
    rp = W.random_periodic(shape=(300, 20, 23), seed=41)
    cs = W.perturbed(W.channel_sphere(shape=(300, 24, 22), center=(40, 12, 11), radius=6,
                                      gx=1e-5), seed=42)
    cs = dataclasses.replace(cs, name=cs.name + " perturbed")
    c3 = W.perturbed(W.cavity3d(shape=(70, 40, 37)), seed=43)
    c2 = W.perturbed(W.cavity2d(shape=(300, 181, 1)), seed=44)
    return [rp, cs, c3, c2]


CASES = slab_cases() + _large_cases()


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_slabs_bitwise_equal_single_domain(oracle_mod, w):
    """Every slab split matches the undivided domain bit for bit, and the fp64 oracle
    (run on the undivided domain) within 1e-6 on the populations and 2e-5 on rho, u, T,
    with the buffer-free swap and (3 slabs) through buffers."""
    n_outer = w.shape[w.dim - 1]
    ref = oracle_states(oracle_mod, w, [7, 8])
    for steps in (7, 8):
        f1, g1, d1 = _single(w, steps)
        counts = sorted({1, 2, 3, n_outer if n_outer <= 13 else 5})   # 1: a ring of one slab
        for k, exchange in [(k, "swap") for k in counts] + [(3, "buffers")]:
            fs, gs, ds, got = _slabs(w, steps, k, chunks=[3, steps - 3], fields=True,
                                     exchange=exchange)
            compare_fields(w, got, ref[steps], tol=TOL_FIELDS, pop_tol=1e-6)
            assert np.array_equal(fs, f1), (steps, k)
            if w.thermal:
                assert np.array_equal(gs, g1), (steps, k)
            assert ds["fluid_cells"] == d1["fluid_cells"]
            assert ds["finite"]
            # the reduction sums chunks of 16 cells in fp32: the slabs chunk the cells
            # differently, so the sums agree to the chunks' rounding (bound: 1e-7 per cell)
            assert abs(ds["mass"] - d1["mass"]) <= 1e-9 * abs(d1["mass"])
            cells = d1["fluid_cells"]
            assert np.allclose(ds["momentum"], d1["momentum"], rtol=0, atol=1e-7 * cells)
            fscale = max(1e-30, float(np.abs(d1["force"]).max()))
            assert np.allclose(ds["force"], d1["force"], rtol=0, atol=1e-5 * fscale)
            if w.thermal:
                hscale = max(1e-30, float(np.abs(d1["heat"]).max()))
                assert np.allclose(ds["heat"], d1["heat"], rtol=0, atol=1e-6 * hscale)
                # the Nusselt numbers, recomputed from the parts' sums with the whole
                # domain's extents, against the library's own on the undivided domain
                assert np.allclose(ds["uT"], d1["uT"], rtol=0, atol=1e-7 * cells)
                for key in ("nu_hot", "nu_cold"):
                    assert abs(ds[key] - d1[key]) <= 1e-5 * max(1.0, abs(d1[key])), key
                assert abs(ds["nu_volume"] - d1["nu_volume"]) <= 1e-3


def test_walls_only_on_the_outer_axis(oracle_mod):
    """Walls (and Dirichlet faces) only at the ends of the outer axis: the end slabs run
    the masked kernels, the inner ones the unmasked kernels."""
    w = outer_walls_case(shape=(64, 20, 24), seed=47)
    ref = oracle_states(oracle_mod, w, [8, 9])
    for steps in (8, 9):
        f1, g1, d1 = _single(w, steps)
        fs, gs, ds, got = _slabs(w, steps, 4, fields=True)
        compare_fields(w, got, ref[steps], tol=TOL_FIELDS, pop_tol=1e-6)
        assert np.abs(fs - f1).max() < 1e-6
        assert np.abs(gs - g1).max() < 1e-6
        assert ds["fluid_cells"] == d1["fluid_cells"]
        assert np.allclose(ds["heat"], d1["heat"], rtol=1e-5, atol=1e-9)


def test_halo_call_order_is_enforced():
    """FILL only at parity 1, DRAIN only at parity 0 after a step, only on HALO sides."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    w = W.random_periodic(shape=(16, 8, 10), seed=46)
    w = dataclasses.replace(w, face_flow=("periodic",) * 4 + ("wall", "halo"))
    sim = Simulation(w)
    nbytes = capi.lbm_halo_bytes(sim.ctx)
    assert nbytes == 4 * 5 * 16 * 8
    buf = torch.empty(nbytes // 4, device="cuda")
    sim.init_equilibrium(*(torch.from_numpy(a).cuda() for a in (w.rho0, w.u0)))
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_pack(sim.ctx, 1, capi.LBM_HALO_DRAIN, buf)   # no step yet
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_pack(sim.ctx, 1, capi.LBM_HALO_FILL, buf)    # parity 0
    sim.step(1)
    capi.lbm_halo_pack(sim.ctx, 1, capi.LBM_HALO_FILL, buf)
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_pack(sim.ctx, 0, capi.LBM_HALO_FILL, buf)    # a WALL side
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_pack(sim.ctx, 2, capi.LBM_HALO_FILL, buf)
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_unpack(sim.ctx, 1, capi.LBM_HALO_DRAIN, buf)  # parity 1
    sim.step(1)
    capi.lbm_halo_unpack(sim.ctx, 1, capi.LBM_HALO_DRAIN, buf)
    torch.cuda.synchronize()
    sim.close()


@pytest.mark.parametrize("w", [W.random_periodic(shape=(40, 12, 9), seed=48),
                               W.perturbed(W.cavity2d(shape=(40, 13, 1)), seed=49)],
                         ids=["periodic ring of one rank", "2-D walled, one rank"])
def test_per_rank_driver_alone(w):
    """The one-slab-per-rank driver with a single rank: a periodic axis makes it a ring with
    itself (its own ghost planes exchanged), a walled one a plain domain."""
    from lattice_boltzmann_cfd_gb300.slabs import DistSlabDomain
    for steps in (6, 7):
        f1, g1, _ = _single(w, steps)
        d = DistSlabDomain(w, 0, 1)
        d.init_equilibrium()
        d.step(steps)
        f, g = d.populations()
        assert np.array_equal(f.cpu().numpy(), f1)
        if w.thermal:
            assert np.array_equal(g.cpu().numpy(), g1)
        d.close()


OVERLAP_CASES = [CASES[i] for i in (0, 3, 5, 7, 8)] + _large_cases()


@pytest.mark.parametrize("w", OVERLAP_CASES, ids=[c.name for c in OVERLAP_CASES])
def test_overlapped_slabs_equal_plain_order(w):
    """The overlapped order (interior planes, boundary planes, exchange on a second stream
    beside the next step's interior) gives the plain order's state bit for bit."""
    n_outer = w.shape[w.dim - 1]
    for steps in (7, 8):
        f1, g1, d1 = _single(w, steps)
        for k in sorted({2, 3, min(n_outer, 5)}):
            from lattice_boltzmann_cfd_gb300.slabs import SlabDomain
            dom = SlabDomain(w, k, overlap=True)
            dom.init_equilibrium()
            for c in (3, steps - 3):
                dom.step(c)
            f, g = dom.populations()
            assert np.array_equal(f.cpu().numpy(), f1), (steps, k)
            if w.thermal:
                assert np.array_equal(g.cpu().numpy(), g1), (steps, k)
            dom.close()


@pytest.mark.parametrize("overlap", [False, True], ids=["plain", "overlap"])
@pytest.mark.parametrize("w", [W.perturbed(W.cavity3d(shape=(70, 40, 37)), seed=43),
                               W.perturbed(W.cavity2d(shape=(300, 181, 1)), seed=44)],
                         ids=["cavity3d 70x40x37", "cavity2d 300x181"])
def test_slabs_200_and_201_steps_against_the_oracle(oracle_mod, w, overlap):
    """Three slabs, 200 and 201 steps, against the oracle on the undivided domain (2e-5 on
    the fields and populations, heat sums 1e-4 relative)."""
    from lattice_boltzmann_cfd_gb300.slabs import SlabDomain
    ref = oracle_states(oracle_mod, w, [200, 201])
    dom = SlabDomain(w, 3, overlap=overlap)
    dom.init_equilibrium()
    done = 0
    for n in (200, 201):
        dom.step(n - done)
        done = n
        f, g = dom.populations()
        rho, u, T = dom.macroscopic()
        got = {"rho": rho.cpu().numpy(), "u": u.cpu().numpy(), "T": T.cpu().numpy(),
               "f": f.cpu().numpy(), "g": g.cpu().numpy()}
        compare_fields(w, got, ref[n])
        assert np.allclose(dom.diagnostics()["heat"], ref[n]["diag"]["heat"], rtol=1e-4,
                           atol=1e-3)
    dom.close()


def test_step_planes_equals_step():
    """lbm_step_planes over any partition of the planes, in any order, is lbm_step(1), at both
    parities; calls that need a whole step are refused while one is partly done."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    cases = [W.perturbed(W.cavity3d(shape=(70, 20, 13)), seed=61),
             W.perturbed(W.cavity2d(shape=(100, 23, 1)), seed=62),
             W.random_periodic(shape=(40, 12, 11), seed=63, lattice=27)]
    rng = np.random.default_rng(9)
    for w in cases:
        n_outer = w.shape[w.dim - 1]
        ref = Simulation(w)
        sim = Simulation(w)
        dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
        for s in (ref, sim):
            s.init_equilibrium(dev(w.rho0), dev(w.u0), dev(w.T_init))
        for step in range(5):
            ref.step(1)
            cuts = sorted(rng.choice(np.arange(1, n_outer), size=3, replace=False))
            parts = list(zip([0] + cuts, cuts + [n_outer]))
            rng.shuffle(parts)
            for i, (lo, hi) in enumerate(parts):
                sim.step_planes(int(lo), int(hi))
                if i < len(parts) - 1:
                    assert sim.parity == step % 2
                    with pytest.raises(capi.LbmError) as e:
                        sim.step(1)
                    assert e.value.status == capi.LBM_ERR_STATE
                    with pytest.raises(capi.LbmError):
                        sim.populations()
                    with pytest.raises(capi.LbmError) as e:
                        sim.step_planes(int(lo), int(hi))        # already stepped
                    assert e.value.status == capi.LBM_ERR_ARG
            assert sim.parity == (step + 1) % 2
            fa, ga = ref.populations()
            fb, gb = sim.populations()
            assert torch.equal(fa, fb), (w.name, step)
            if w.thermal:
                assert torch.equal(ga, gb), (w.name, step)
        with pytest.raises(capi.LbmError):
            sim.step_planes(0, n_outer + 1)
        with pytest.raises(capi.LbmError):
            sim.step_planes(3, 3)
        ref.close()
        sim.close()
    two = Simulation(W.random_periodic(shape=(16, 8, 6), seed=64), streaming="pull")
    w2 = W.random_periodic(shape=(16, 8, 6), seed=64)
    two.init_equilibrium(*(torch.from_numpy(a).cuda() for a in (w2.rho0, w2.u0)))
    with pytest.raises(capi.LbmError) as e:
        two.step_planes(0, 6)
    assert e.value.status == capi.LBM_ERR_UNSUPPORTED
    two.close()
