"""Block partitioning on the host (CPU): the cut of the domain into blocks and the routing of
the per-axis halo exchange between torch.distributed ranks (gloo).

Each rank stands in for one block: its pack stamps (rank, axis, side, phase) into the buffer
and its unpack records what arrived.  Along every split axis a block's low side faces its
low neighbour's high side (wrapping on a periodic axis), the axes run z, then y, then x,
and the ends of a walled axis receive nothing."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from lattice_boltzmann_cfd_gb300 import workloads as W  # noqa: E402
from lattice_boltzmann_cfd_gb300.blocks import (block_counts, block_index,  # noqa: E402
                                                block_neighbours, block_part, owned_slices)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _stamp(rank, axis, side, phase):
    return 1000.0 * rank + 100.0 * axis + 10.0 * side + phase


def _worker(rank, world, port, nb, periodic, dim, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.blocks import block_exchange
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = []
    send = [[torch.zeros(5), torch.zeros(5)] for _ in range(3)]
    recv = [[torch.full((5,), -1.0), torch.full((5,), -1.0)] for _ in range(3)]
    pack = lambda a, side, phase, buf: buf.fill_(_stamp(rank, a, side, phase))
    unpack = lambda a, side, phase, buf: got.append((a, side, phase, buf.tolist()))
    for phase in (0, 1, 0):
        block_exchange(rank, nb, periodic, dim, phase, pack, unpack, send, recv)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def _expected(rank, nb, periodic, dim):
    nbs = block_neighbours(rank, nb, periodic)
    exp = []
    for phase in (0, 1, 0):
        for a in range(dim - 1, -1, -1):
            if nb[a] < 2:
                continue
            for side in (0, 1):
                if nbs[a][side] is not None:
                    exp.append((a, side, phase, [_stamp(nbs[a][side], a, 1 - side, phase)] * 5))
    return exp


@pytest.mark.parametrize("nb,periodic,dim", [
    ((2, 2, 1), (True, True, True), 3),
    ((2, 2, 1), (False, True, True), 3),
    ((1, 2, 2), (True, False, False), 3),
    ((2, 1, 2), (True, True, True), 3),
    ((2, 2, 1), (True, False, False), 2),
    ((3, 1, 1), (False, True, True), 2),
])
def test_block_exchange_routes_each_face(nb, periodic, dim):
    import multiprocessing as mp
    world = nb[0] * nb[1] * nb[2]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, nb, periodic, dim, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            assert out[r] == _expected(r, nb, periodic, dim), r


def test_block_neighbours_wrap_and_stop():
    nb = (3, 2, 1)
    per = (True, False, False)
    # block (0, 1, 0): x wraps to block 2, y has no high neighbour
    b = block_index((0, 1, 0), nb)
    nbs = block_neighbours(b, nb, per)
    assert nbs[0] == (block_index((2, 1, 0), nb), block_index((1, 1, 0), nb))
    assert nbs[1] == (block_index((0, 0, 0), nb), None)
    assert nbs[2] == (None, None)


@pytest.mark.parametrize("parts,shape,dim,want", [
    (4, (64, 64, 1), 2, (2, 2, 1)),
    (8, (64, 64, 1), 2, (2, 4, 1)),      # the outer axis takes the larger count
    (8, (64, 64, 64), 3, (1, 2, 4)),     # x rows kept whole; z takes the larger count
    (4, (64, 64, 64), 3, (1, 2, 2)),
    (2, (64, 64, 64), 3, (1, 1, 2)),
    (6, (96, 64, 32), 3, (1, 3, 2)),     # closest to cubes among the y-z splits
    (3, (5, 2, 2), 3, (3, 1, 1)),        # only x has room for three
    (4, (64, 2, 1), 3, (4, 1, 1)),       # y and z too thin: x takes the pieces
])
def test_block_counts(parts, shape, dim, want):
    assert block_counts(shape, dim, parts) == want


def test_block_counts_rejects_too_many():
    with pytest.raises(ValueError):
        block_counts((2, 2, 1), 2, 5)


@pytest.mark.parametrize("nb", [(2, 2, 1), (1, 3, 2), (3, 2, 2), (7, 1, 1)])
def test_block_parts_tile_the_domain(nb):
    """The owned cells of the blocks cover every cell of the domain once, with the fields
    of those cells; a split walled axis keeps its walls at the end blocks, a split periodic
    one gets HALO faces everywhere."""
    w = W.perturbed(W.cavity3d(shape=(7, 6, 5)), seed=3)
    seen = np.zeros(w.grid, int)
    for b in range(nb[0] * nb[1] * nb[2]):
        local, sides, coords = block_part(w, nb, b)
        own = owned_slices(sides, coords)
        sel = np.ix_(*(np.array(coords[a])[own[2 - a]] for a in (2, 1, 0)))
        seen[sel] += 1
        assert np.array_equal(local.rho0[own], w.rho0[sel])
        assert np.array_equal(local.T_init[own], w.T_init[sel])
        assert np.array_equal(local.u0[(slice(None),) + own], w.u0[(slice(None),) + sel])
        for a in range(3):
            low, high = sides[a]
            assert local.face_flow[2 * a] == ("halo" if low else w.face_flow[2 * a])
            assert local.face_flow[2 * a + 1] == ("halo" if high else w.face_flow[2 * a + 1])
            assert local.shape[a] == len(coords[a])
    assert (seen == 1).all()
    wp = W.random_periodic(shape=(6, 6, 6), seed=4)
    local, sides, _ = block_part(wp, (2, 1, 3), 0)
    assert sides[0] == (True, True) and sides[1] == (False, False) and sides[2] == (True, True)
    assert local.face_flow == ("halo", "halo", "periodic", "periodic", "halo", "halo")


def _dying_block(rank, world, port, out):
    import datetime
    import time
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.blocks import block_exchange
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=8))
    dist.barrier()
    if rank == 3:
        os._exit(0)                  # leaves between steps: no exchange in flight
    send = [[torch.zeros(4), torch.zeros(4)] for _ in range(3)]
    recv = [[torch.zeros(4), torch.zeros(4)] for _ in range(3)]
    t0 = time.time()
    try:
        block_exchange(rank, (2, 2, 1), (True, True, True), 3, 0,
                       lambda a, s, p, b: b.fill_(1.0), lambda a, s, p, b: None, send, recv)
        out[rank] = ("completed", 0.0)
    except Exception as e:           # the back-end reports the lost peer
        out[rank] = (type(e).__name__, time.time() - t0)


def test_lost_block_fails_its_neighbours_next_exchange():
    """In a 2 x 2 split, a rank that leaves between steps makes the exchange of each block
    that faces it (along y, then along x) raise instead of waiting forever."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_dying_block, args=(r, 4, port, out)) for r in range(4)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        # blocks 1 (x-neighbour of 3) and 2 (y-neighbour of 3) face the lost rank
        for r in (1, 2):
            kind, seconds = out[r]
            assert kind != "completed", r
            assert seconds < 30


def _diag_worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.slabs import allreduce_diagnostics
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = allreduce_diagnostics(_diag_case(), _fake_diag(rank))
    dist.barrier()
    dist.destroy_process_group()


def _diag_case():
    return W.cavity3d(shape=(12, 10, 8))


def _fake_diag(rank):
    rng = np.random.default_rng(100 + rank)
    return {"mass": float(rng.uniform(10, 20)), "momentum": list(rng.normal(size=3)),
            "force": list(rng.normal(size=3)), "heat": list(rng.normal(size=6)),
            "uT": list(rng.normal(size=3)), "fluid_cells": int(rng.integers(100, 200)),
            "finite": rank != 2}


def test_allreduce_diagnostics_sums_every_rank():
    """The all-reduce of the ranks' sums (gloo, 3 ranks) equals combine_diagnostics of the
    summed parts; one rank with a non-finite state makes the whole not finite; the Nusselt
    numbers follow the whole domain's extents (the cavity's hot x = 0 and cold x = L faces)."""
    import multiprocessing as mp
    from lattice_boltzmann_cfd_gb300.slabs import combine_diagnostics, diag_vector
    world = 3
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_diag_worker, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        want = combine_diagnostics(
            _diag_case(), list(np.sum([diag_vector(_fake_diag(r)) for r in range(world)],
                                      axis=0)))
        for r in range(world):
            got = out[r]
            assert got["fluid_cells"] == want["fluid_cells"]
            assert got["finite"] is False
            for key in ("mass", "nu_hot", "nu_cold", "nu_volume"):
                assert got[key] == pytest.approx(want[key], rel=1e-12, abs=1e-12), key
            for key in ("momentum", "force", "heat", "uT"):
                assert np.allclose(got[key], want[key], rtol=1e-12, atol=1e-12), key
    # the wall heat of the hot face (x = 0, face 0) over the whole face: |heat| H / (dT A)
    w = _diag_case()
    heat0 = sum(_fake_diag(r)["heat"][0] for r in range(world))
    assert want["nu_hot"] == pytest.approx(abs(heat0) * 12 / (1.0 * 10 * 8), rel=1e-12)


@pytest.mark.parametrize("nb", [(2, 2, 1), (1, 3, 2), (3, 2, 2)])
def test_part_of_takes_a_parts_cells(nb):
    """part_of cuts a whole-domain field at a part's coordinates, ghost planes included, as
    block_part cuts the initial fields."""
    from lattice_boltzmann_cfd_gb300.slabs import part_of
    w = W.perturbed(W.cavity3d(shape=(7, 6, 5)), seed=5)
    for b in range(nb[0] * nb[1] * nb[2]):
        local, _, coords = block_part(w, nb, b)
        assert np.array_equal(part_of(torch.from_numpy(w.rho0), coords, lead=0).numpy(),
                              local.rho0)
        assert np.array_equal(part_of(torch.from_numpy(w.u0), coords).numpy(), local.u0)
