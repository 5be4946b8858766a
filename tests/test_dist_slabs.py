"""Routing of the slab halo exchange between torch.distributed ranks (gloo, on the CPU).

Each rank stands in for one slab: its pack stamps (rank, side, phase) into the buffer and its
unpack records what arrived.  Slab r's low side faces slab r-1's high side (slab 0's low
side faces the last slab's high side when the outer axis is periodic); every inner face must
receive exactly the opposite side's buffer of its neighbour, in the same phase, and the end
faces of a walled axis nothing.  The two-rank ring, where both neighbours are one rank,
checks that messages pair by side and not by arrival order."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _stamp(rank, side, phase):
    return 100.0 * rank + 10.0 * side + phase


def _worker(rank, world, port, periodic, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.slabs import ring_exchange
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = []
    send = [torch.zeros(6), torch.zeros(6)]
    recv = [torch.full((6,), -1.0), torch.full((6,), -1.0)]
    pack = lambda side, phase, buf: buf.fill_(_stamp(rank, side, phase))
    unpack = lambda side, phase, buf: got.append((side, phase, buf.tolist()))
    syncs = []
    for phase in (0, 1, 0, 1):
        ring_exchange(rank, world, periodic, phase, pack, unpack, send, recv,
                      sync=lambda: syncs.append(1))
    out[rank] = (got, len(syncs))
    dist.barrier()
    dist.destroy_process_group()


def _expected(rank, world, periodic):
    lo = rank - 1 if rank > 0 else (world - 1 if periodic else None)
    hi = rank + 1 if rank < world - 1 else (0 if periodic else None)
    exp = []
    for phase in (0, 1, 0, 1):
        for side, nb in ((0, lo), (1, hi)):
            if nb is not None:
                exp.append((side, phase, [_stamp(nb, 1 - side, phase)] * 6))
    return exp


@pytest.mark.parametrize("world,periodic", [(2, True), (2, False), (3, True), (3, False)])
def test_ring_exchange_routes_each_face(world, periodic):
    import torch.multiprocessing as mp
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, periodic, out), nprocs=world, join=True)
    for r in range(world):
        got, nsync = out[r]
        assert got == _expected(r, world, periodic), r
        assert nsync == 2 * 4


def test_ring_of_one_slab_crosses_its_own_buffers():
    from lattice_boltzmann_cfd_gb300.slabs import ring_exchange
    got = []
    send = [torch.zeros(3), torch.zeros(3)]
    ring_exchange(0, 1, True, 1, lambda s, p, b: b.fill_(_stamp(0, s, p)),
                  lambda s, p, b: got.append((s, b[0].item())), send, None)
    assert got == [(0, _stamp(0, 1, 1)), (1, _stamp(0, 0, 1))]
    got.clear()
    ring_exchange(0, 1, False, 1, lambda s, p, b: b.fill_(1.0),
                  lambda s, p, b: got.append(s), send, None)
    assert got == []


def test_slab_parts_tile_the_domain():
    """The slabs' owned planes cover the outer axis once; ghost planes are the neighbours'
    boundary planes (wrapped on a periodic axis); inner faces become HALO faces."""
    import numpy as np
    from lattice_boltzmann_cfd_gb300 import workloads as W
    from lattice_boltzmann_cfd_gb300.slabs import slab_part
    for w in (W.random_periodic(shape=(5, 4, 11), seed=1), W.cavity3d(shape=(5, 4, 11)),
              W.cavity2d(shape=(6, 9, 1))):
        axis = w.dim - 1
        n = w.shape[axis]
        periodic = w.face_flow[2 * axis] == "periodic"
        for k in (1, 2, 3, n):
            owned = []
            for r in range(k):
                local, (low, high), planes = slab_part(w, k, r)
                inner = planes[(1 if low else 0):len(planes) - (1 if high else 0)]
                owned += inner
                assert local.shape[axis] == len(planes)
                if low:
                    assert planes[0] == (inner[0] - 1) % n
                    assert local.face_flow[2 * axis] == "halo"
                else:
                    assert local.face_flow[2 * axis] == w.face_flow[2 * axis]
                if high:
                    assert planes[-1] == (inner[-1] + 1) % n
                assert (low and high) or not periodic
                np_axis = 0 if w.dim == 3 else 1
                assert np.array_equal(local.rho0, np.take(w.rho0, planes, axis=np_axis))
            assert owned == list(range(n))


def _dying_worker(rank, world, port, out):
    import datetime
    import time
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.slabs import ring_exchange
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=8))
    dist.barrier()
    if rank == 1:
        os._exit(0)                  # leaves between steps: no exchange in flight
    send = [torch.zeros(4), torch.zeros(4)]
    recv = [torch.zeros(4), torch.zeros(4)]
    t0 = time.time()
    try:
        ring_exchange(0, 2, True, 0, lambda s, p, b: b.fill_(1.0), lambda s, p, b: None,
                      send, recv)
        out[0] = ("completed", 0.0)
    except Exception as e:           # the back-end reports the lost peer
        out[0] = (type(e).__name__, time.time() - t0)


def test_lost_rank_fails_the_next_exchange():
    """A rank that leaves between steps makes its neighbour's next halo exchange raise (a
    lost connection, or the process group's timeout) instead of waiting forever."""
    import torch.multiprocessing as mp
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_dying_worker, args=(2, port, out), nprocs=2, join=True)
    kind, seconds = out[0]
    assert kind != "completed"
    assert seconds < 30
