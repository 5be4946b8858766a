"""JobPipeline (host-link copies overlapped with the neighbouring jobs' steps) against the
same jobs run one after another: every job's outputs and diagnostics are bit-identical,
with the copies in one piece and cut into one piece per step."""
import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _pinned(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


@pytest.mark.parametrize("make", [lambda s: W.perturbed(W.cavity3d(shape=(48, 20, 18)), seed=s),
                                  lambda s: W.random_periodic(shape=(64, 24, 20), seed=s),
                                  lambda s: W.perturbed(W.cavity2d(shape=(96, 80, 1)), seed=s)],
                         ids=["cavity3d", "periodic", "cavity2d"])
@pytest.mark.parametrize("piece_bytes", [32 << 20, 4096], ids=["whole", "pieces"])
@pytest.mark.parametrize("steps", [9, 1, 0])
@pytest.mark.parametrize("overlap_readout", [False, True], ids=["readout_alone", "readout_overlap"])
def test_pipeline_matches_serial_jobs(make, piece_bytes, steps, overlap_readout):
    from lattice_boltzmann_cfd_gb300 import Simulation
    from lattice_boltzmann_cfd_gb300.pipeline import JobPipeline
    ws = [make(seed) for seed in (3, 4, 5, 6, 7)]
    jobs = []
    for w in ws:
        ins = tuple(_pinned(a) for a in (w.rho0, w.u0, w.T_init if w.thermal else None))
        outs = tuple(None if t is None else torch.empty_like(t).pin_memory() for t in ins)
        jobs.append((ins, outs))
    # one after another, on device buffers
    sim = Simulation(ws[0])
    serial = []
    for (ins, _), w in zip(jobs, ws):
        dev = [None if t is None else t.cuda() for t in ins]
        sim.init_equilibrium(*dev)
        sim.step(steps)
        rho, u, T = sim.macroscopic()
        serial.append(([t.cpu() for t in (rho, u) + ((T,) if T is not None else ())],
                       sim.diagnostics()))
    sim.close()
    # pipelined
    sim = Simulation(ws[0])
    diags = JobPipeline(sim, piece_bytes=piece_bytes,
                        overlap_readout=overlap_readout).run(jobs, steps)
    sim.close()
    for (fields, d), (_, outs), dp in zip(serial, jobs, diags):
        for a, b in zip(fields, [t for t in outs if t is not None]):
            assert torch.equal(a, b)
        for key in ("mass", "momentum", "heat", "fluid_cells", "uT"):
            assert d[key] == dp[key], key


def test_pipeline_without_readout():
    """Jobs whose outputs are None run and return diagnostics only."""
    from lattice_boltzmann_cfd_gb300 import Simulation
    from lattice_boltzmann_cfd_gb300.pipeline import JobPipeline
    w = W.random_periodic(shape=(32, 16, 16), seed=9)
    ins = (_pinned(w.rho0), _pinned(w.u0), None)
    sim = Simulation(w)
    for piece_bytes in (32 << 20, 1000):
        diags = JobPipeline(sim, piece_bytes=piece_bytes).run([(ins, None)] * 3, 4)
        assert len(diags) == 3 and diags[0]["mass"] == diags[2]["mass"]
    sim.close()


def test_ib_block_search_returns_the_fastest_candidate():
    """The measured search of the immersed-boundary block edge times every candidate and
    returns the one with the lowest step time."""
    from lattice_boltzmann_cfd_gb300.tuning import default_candidates, search_ib_block
    w = W.channel_ib_sphere(shape=(64, 48, 48), center=(20.3, 23.7, 24.2), radius=8)
    cands = default_candidates(w)
    assert cands[0] == 2 and cands[-1] == 16
    best, times = search_ib_block(w, candidates=[2, 4, 8], steps=8, warmup=2)
    assert set(times) == {2, 4, 8} and all(t > 0 for t in times.values())
    assert times[best] == min(times.values())


def test_two_pipelines_on_one_simulation():
    """A pipeline built later on the same simulation moves it to its own stream; each run()
    takes the simulation back, so runs of either pipeline, in any order, stay correct."""
    from lattice_boltzmann_cfd_gb300 import Simulation
    from lattice_boltzmann_cfd_gb300.pipeline import JobPipeline
    ws = [W.random_periodic(shape=(64, 24, 20), seed=s) for s in (11, 12)]
    jobs = []
    for w in ws:
        ins = (_pinned(w.rho0), _pinned(w.u0), None)
        jobs.append((ins, tuple(None if t is None else torch.empty_like(t).pin_memory()
                                for t in ins)))
    sim = Simulation(ws[0])
    want = []
    for (ins, _) in jobs:
        sim.init_equilibrium(*[None if t is None else t.cuda() for t in ins])
        sim.step(7)
        rho, u, _ = sim.macroscopic()
        torch.cuda.synchronize()
        want.append((rho.cpu(), u.cpu()))
    a = JobPipeline(sim, piece_bytes=4096)
    b = JobPipeline(sim, overlap_readout=True)
    for pipe in (a, b, a):
        for t in (o for _, outs in jobs for o in outs if o is not None):
            t.fill_(float("nan"))
        pipe.run(jobs, 7)
        for (rho, u), (_, outs) in zip(want, jobs):
            assert torch.equal(rho, outs[0]) and torch.equal(u, outs[1])
    sim.close()
