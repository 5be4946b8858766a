"""The one-slab-per-rank driver with two ranks, on the GPU through the C ABI.

Two torch.distributed ranks (gloo, one process each) share the one GPU of the test box:
each steps its slab with the library and exchanges halos through page-locked host buffers,
which the halo kernels write and read directly, so no kernel ever waits for the other
rank (the waiting is on the host, in the gloo messages).  The gathered owned planes must
equal the undivided domain bit for bit and match the fp64 oracle, with the plain order and
with the overlapped one, for a periodic ring (both neighbours are the other rank) and for
walled ends in 3-D and 2-D.
"""
import datetime
import os
import socket

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W
from parity_util import compare_fields, oracle_states

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STEPS = (7, 8)


def _case(name):
    if name == "periodic ring":
        return W.random_periodic(shape=(40, 12, 20), seed=71)
    if name == "cavity3d walled":
        return W.perturbed(W.cavity3d(shape=(36, 20, 22)), seed=72)
    return W.perturbed(W.cavity2d(shape=(70, 30, 1)), seed=73)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, name, overlap, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.slabs import DistSlabDomain
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=120))
    w = _case(name)
    d = DistSlabDomain(w, rank, world, device="cuda:0", transport="host", overlap=overlap)
    d.init_equilibrium()
    res, done = {}, 0
    for n in STEPS:
        d.step(n - done)
        done = n
        f, g = d.populations()
        res[n] = (f.cpu().numpy(), None if g is None else g.cpu().numpy())
    res["diag"] = d.global_diagnostics()      # a collective: every rank calls it
    out[rank] = res
    d.close()
    dist.barrier()
    dist.destroy_process_group()


def _single(w, steps):
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    sim = Simulation(w)
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sim.init_equilibrium(dev(w.rho0), dev(w.u0), dev(w.T_init))
    sim.step(steps)
    f, g = sim.populations()
    out = (f.cpu().numpy(), None if g is None else g.cpu().numpy())
    sim.close()
    return out


@pytest.mark.parametrize("overlap", [False, True], ids=["plain", "overlap"])
@pytest.mark.parametrize("name", ["periodic ring", "cavity3d walled", "cavity2d walled"])
def test_two_ranks_share_the_gpu(oracle_mod, name, overlap):
    import torch.multiprocessing as mp
    assert torch.cuda.is_available(), "CUDA device required"
    w = _case(name)
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.spawn(_rank, args=(2, _free_port(), name, overlap, out), nprocs=2, join=True)
    ax = 1 if w.dim == 3 else 2      # outer axis of a (Q, nz, ny, nx) population array
    ref = oracle_states(oracle_mod, w, list(STEPS))
    for n in STEPS:
        f = np.concatenate([out[r][n][0] for r in range(2)], axis=ax)
        g = np.concatenate([out[r][n][1] for r in range(2)], axis=ax) if w.thermal else None
        f1, g1 = _single(w, n)
        assert np.array_equal(f, f1), n
        if w.thermal:
            assert np.array_equal(g, g1), n
        fluid = np.ones(w.grid, bool)
        assert np.abs(f - ref[n]["f"])[:, fluid].max() <= 1e-6
        if w.thermal:
            assert np.abs(g - ref[n]["g"])[:, fluid].max() <= 1e-6
    # the all-reduced diagnostics after the last step, against the undivided domain's
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    sim = Simulation(w)
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sim.init_equilibrium(dev(w.rho0), dev(w.u0), dev(w.T_init))
    sim.step(STEPS[-1])
    d1 = sim.diagnostics()
    sim.close()
    for r in range(2):
        dg = out[r]["diag"]
        assert dg["fluid_cells"] == d1["fluid_cells"] and dg["finite"]
        assert abs(dg["mass"] - d1["mass"]) <= 1e-9 * abs(d1["mass"])
        if w.thermal:
            for key in ("nu_hot", "nu_cold"):
                assert abs(dg[key] - d1[key]) <= 1e-5 * max(1.0, abs(d1[key])), key
            assert abs(dg["nu_volume"] - d1["nu_volume"]) <= 1e-3
