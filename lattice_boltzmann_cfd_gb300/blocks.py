"""A domain cut into blocks along several axes: one library context per block, with the
per-axis halo exchange driven from the host (the block partitioning of "Multi-GPU thermal
lattice Boltzmann simulations using OpenACC and MPI", Sec. 4, Fig. 5).

Each block has a ghost plane at every face it shares with another block.  The exchange runs
axis by axis (z, then y, then x), with the whole plane of an axis moved, the ghost rows of
the other axes included, so that the populations of diagonal links reach the block across
an edge or a corner through the block beside it (lbm_halo_axis_pack / _unpack, or
lbm_halo_axis_swap_many between blocks on one device).  BlockDomain holds every block in one
process; DistBlockDomain is one block per torch.distributed rank.  The slabs of slabs.py are
the one-axis case; the helpers shared with them (field splitting, whole-domain diagnostics,
checkpoints, point-to-point messages) live there.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import capi
from .slabs import (_as_tensor, _device_index, allreduce_diagnostics, combine_diagnostics,
                    diag_vector, halo_messages, part_of, split_ranges)
from .solver import Simulation


def block_counts(shape, dim: int, parts: int):
    """(bx, by, bz) with bx * by * bz = parts, following the pages' two rules: keep the rows
    along x (the contiguous axis) whole where possible, and make the block extents as even
    as possible.  In 3-D, x is split only when y and z cannot take every piece; among the
    remaining splits the one whose blocks are closest to cubes (the smallest largest-to-
    smallest extent ratio) wins, the outer axis taking the larger count on a tie.  A 2-D
    domain cut into blocks is cut along x and y."""
    best = None
    for bz in (range(1, parts + 1) if dim == 3 else (1,)):
        if parts % bz:
            continue
        for by in range(1, parts // bz + 1):
            if (parts // bz) % by:
                continue
            bx = parts // (bz * by)
            nb = (bx, by, bz)
            if any(nb[a] > shape[a] for a in range(3)):
                continue
            ext = [shape[a] / nb[a] for a in range(dim)]
            key = (dim == 3 and bx > 1, max(ext) / min(ext), -nb[dim - 1],
                   -nb[1 if dim == 3 else 0])
            if best is None or key < best[0]:
                best = (key, nb)
    if best is None:
        raise ValueError(f"{parts} blocks do not fit the grid {tuple(shape)}")
    return best[1]


def block_index(bi, nb) -> int:
    """Rank (or list position) of block bi = (i, j, k): x fastest."""
    return bi[0] + nb[0] * (bi[1] + nb[1] * bi[2])


def block_coords(b: int, nb):
    return (b % nb[0], (b // nb[0]) % nb[1], b // (nb[0] * nb[1]))


def block_part(w, nb, b: int):
    """Block b of ``w`` cut into nb = (bx, by, bz) pieces: (local workload, per-axis (low,
    high) ghost flags, per-axis list of the domain coordinate of each local plane).  An axis
    split into two or more pieces gets ghost planes at its inner faces, and at both ends
    when it is periodic (the pieces form a ring); its end blocks keep a wall face."""
    if getattr(w, "ib_x", None) is not None and len(w.ib_x):
        raise ValueError("blocks do not take immersed-boundary samples")
    bi = block_coords(b, nb)
    faces = list(w.face_flow)
    shape = list(w.shape)
    sides, coords = [], []
    for a in range(3):
        n = w.shape[a]
        split = a < w.dim and nb[a] > 1
        if a >= w.dim and nb[a] != 1:
            raise ValueError("a 2-D domain has one block along z")
        if split and nb[a] > n:
            raise ValueError("more blocks than planes along an axis")
        periodic = w.face_flow[2 * a] == "periodic"
        lo, hi = split_ranges(n, nb[a])[bi[a]] if split else (0, n)
        low = split and (periodic or bi[a] > 0)
        high = split and (periodic or bi[a] < nb[a] - 1)
        planes = ([(lo - 1) % n] if low else []) + list(range(lo, hi)) + \
                 ([hi % n] if high else [])
        if low:
            faces[2 * a] = "halo"
        if high:
            faces[2 * a + 1] = "halo"
        shape[a] = len(planes)
        sides.append((low, high))
        coords.append(planes)
    sel = np.ix_(coords[2], coords[1], coords[0])     # fields are (nz, ny, nx)

    def take(a, lead=0):
        if a is None:
            return None
        return np.ascontiguousarray(a[(slice(None),) * lead + sel])

    local = dataclasses.replace(
        w, shape=tuple(shape), face_flow=tuple(faces), solid=take(w.solid),
        rho0=take(w.rho0), u0=take(w.u0, 1), T_init=take(w.T_init))
    return local, sides, coords


def block_neighbours(b: int, nb, periodic):
    """Per axis, the (low, high) neighbour block indices of block b (None at the end of a
    walled axis or along an axis that is not split).  periodic: per axis."""
    bi = block_coords(b, nb)
    out = []
    for a in range(3):
        if nb[a] < 2:
            out.append((None, None))
            continue
        nbs = []
        for d in (-1, 1):
            j = list(bi)
            j[a] += d
            if 0 <= j[a] < nb[a]:
                nbs.append(block_index(j, nb))
            elif periodic[a]:
                j[a] %= nb[a]
                nbs.append(block_index(j, nb))
            else:
                nbs.append(None)
        out.append(tuple(nbs))
    return out


def exchange_axes(dim: int, nb):
    """The axes a block exchange runs through, in order: z, y, x, those split only."""
    return [a for a in range(dim - 1, -1, -1) if nb[a] > 1]


def block_groups(ext, sides, dim: int):
    """(interior box or None, [boundary boxes]) of a block with local extents ext (x, y, z)
    and per-axis (low, high) ghost flags: the boundary is every cell within two planes of a
    HALO face (its ghost plane and the first owned plane), cut into disjoint boxes axis by
    axis (z, then y, then x); the interior is the rest.  Boxes are (lo, hi) triples of cell
    coordinates.  A block too thin for an interior is one boundary box."""
    lo = [0, 0, 0]
    hi = [int(ext[0]), int(ext[1]), int(ext[2]) if dim == 3 else 1]
    inner_lo = [2 if sides[a][0] else 0 for a in range(3)]
    inner_hi = [hi[a] - 2 if sides[a][1] else hi[a] for a in range(3)]
    if any(inner_hi[a] <= inner_lo[a] for a in range(3)):
        return None, [(tuple(lo), tuple(hi))]
    boundary = []
    for a in range(dim - 1, -1, -1):
        if inner_lo[a] > lo[a]:
            b_hi = list(hi)
            b_hi[a] = inner_lo[a]
            boundary.append((tuple(lo), tuple(b_hi)))
            lo[a] = inner_lo[a]
        if inner_hi[a] < hi[a]:
            b_lo = list(lo)
            b_lo[a] = inner_hi[a]
            boundary.append((tuple(b_lo), tuple(hi)))
            hi[a] = inner_hi[a]
    return (tuple(lo), tuple(hi)), boundary


def block_exchange(b: int, nb, periodic, dim: int, phase: int, pack, unpack, send, recv,
                   group=None, sync=None):
    """One halo exchange of block ``b`` (its torch.distributed rank) with its neighbours:
    per axis in exchange_axes order, the packs, the messages (halo_messages), then the
    unpacks, before the next axis starts.  pack(axis, side, phase, buf) fills
    send[axis][side]; unpack(axis, side, phase, buf) consumes a buffer; sync(), if given,
    runs after each axis's packs and after its receives."""
    nbs = block_neighbours(b, nb, periodic)
    for a in exchange_axes(dim, nb):
        for side in (0, 1):
            if nbs[a][side] is not None:
                pack(a, side, phase, send[a][side])
        if sync is not None:
            sync()
        arrived = halo_messages(nbs[a], send[a], recv[a], group)
        if sync is not None:
            sync()
        for side, buf in arrived:
            unpack(a, side, phase, buf)


def owned_slices(sides, coords, lead=0):
    """Index of a block's owned cells in a local field with ``lead`` leading axes."""
    idx = [slice(None)] * lead
    for a in (2, 1, 0):
        low, high = sides[a]
        idx.append(slice(1 if low else 0, len(coords[a]) - (1 if high else 0)))
    return tuple(idx)


class BlockDomain:
    """The workload ``w`` cut into nb = (bx, by, bz) blocks (block_counts picks nb for a
    number of pieces), block b on ``devices[b % len(devices)]``, all driven from this
    process.  Each step is followed by the exchange of every split axis, z then y then x;
    between steps every owned cell holds what one undivided domain would hold.

    ``exchange``: "swap" moves each face with one buffer-free kernel (lbm_halo_axis_swap,
    blocks on one device), "buffers" packs, copies and unpacks; "auto" takes the swap on one
    device.  ``overlap``: see step (one device only)."""

    def __init__(self, w, nb, devices=None, exchange: str = "auto", overlap: bool = False):
        import torch
        if exchange not in ("auto", "swap", "buffers"):
            raise ValueError("exchange must be 'auto', 'swap' or 'buffers'")
        nb = tuple(int(v) for v in nb)
        if len(nb) != 3 or min(nb) < 1:
            raise ValueError("nb must be three positive block counts")
        self.w, self.nb, self.dim = w, nb, w.dim
        self.periodic = [w.face_flow[2 * a] == "periodic" for a in range(3)]
        devices = list(devices) if devices else [torch.device("cuda")]
        nblocks = nb[0] * nb[1] * nb[2]
        self.multi_device = len({_device_index(d) for d in devices[:nblocks]}) > 1
        if exchange == "swap" and self.multi_device:
            raise ValueError("the buffer-free swap needs every block on one device")
        self.swap = exchange == "swap" or (exchange == "auto" and not self.multi_device)
        self.blocks, self.sides, self.coords, self.buffers = [], [], [], []
        self.face_floats = []     # per block and axis: floats of one face's buffer
        for b in range(nblocks):
            local, sides, coords = block_part(w, nb, b)
            sim = Simulation(local, device=devices[b % len(devices)])
            bufs, floats = [], []
            for a in range(3):
                nfloat = capi.lbm_halo_axis_bytes(sim.ctx, a) // 4 if (
                    a < w.dim and nb[a] > 1) else 0
                floats.append(nfloat)
                bufs.append([torch.empty(nfloat, dtype=torch.float32, device=sim.device)
                             for _ in range(2)] if nfloat and not self.swap else None)
            self.blocks.append(sim)
            self.sides.append(sides)
            self.coords.append(coords)
            self.buffers.append(bufs)
            self.face_floats.append(floats)
        self.overlap = bool(overlap)
        if self.overlap and self.multi_device:
            raise ValueError("overlap needs every block on one device")
        self.groups = [block_groups([len(c) for c in coords], sides, w.dim)
                       for coords, sides in zip(self.coords, self.sides)]
        dev = self.blocks[0].device
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev) if self.overlap else None
        self._pending = None    # event: the last exchange's unpacks are queued before it

    @property
    def parity(self) -> int:
        return self.blocks[0].parity

    def pairs(self, a: int):
        """(block, its high neighbour along axis a) for every face between blocks."""
        out = []
        for b in range(len(self.blocks)):
            hi = block_neighbours(b, self.nb, self.periodic)[a][1]
            if hi is not None:
                out.append((b, hi))
        return out

    def _sync(self):
        import torch
        if self.multi_device:
            for d in {s.device for s in self.blocks}:
                torch.cuda.synchronize(d)

    def _exchange(self, phase: int):
        for a in exchange_axes(self.dim, self.nb):
            pairs = self.pairs(a)
            if self.swap:     # every face of the axis in one launch (32 per launch at most)
                for k in range(0, len(pairs), 32):
                    chunk = pairs[k:k + 32]
                    capi.lbm_halo_axis_swap_many([self.blocks[lo].ctx for lo, _ in chunk],
                                                 [self.blocks[hi].ctx for _, hi in chunk],
                                                 a, phase)
                continue
            for lo, hi in pairs:
                capi.lbm_halo_axis_pack(self.blocks[lo].ctx, a, 1, phase, self.buffers[lo][a][1])
                capi.lbm_halo_axis_pack(self.blocks[hi].ctx, a, 0, phase, self.buffers[hi][a][0])
            self._sync()
            for lo, hi in pairs:
                to_lo = self.buffers[hi][a][0].to(self.blocks[lo].device)
                to_hi = self.buffers[lo][a][1].to(self.blocks[hi].device)
                capi.lbm_halo_axis_unpack(self.blocks[lo].ctx, a, 1, phase, to_lo)
                capi.lbm_halo_axis_unpack(self.blocks[hi].ctx, a, 0, phase, to_hi)
            self._sync()

    def init_equilibrium(self):
        """Every block from the workload's initial fields (its ghost planes included)."""
        import torch
        for sim, coords in zip(self.blocks, self.coords):
            sel = np.ix_(coords[2], coords[1], coords[0])

            def dev(a, lead=0):
                if a is None:
                    return None
                t = np.ascontiguousarray(a[(slice(None),) * lead + sel])
                return torch.from_numpy(t).to(sim.device)
            sim.init_equilibrium(dev(self.w.rho0), dev(self.w.u0, 1), dev(self.w.T_init))

    def step(self, n: int = 1):
        """n time steps, each followed by its exchange (FILL after even, DRAIN after odd).
        With ``overlap``: each block's interior box, a wait for the previous exchange, its
        boundary boxes, then the exchange on a second stream beside the next step's interior
        (block_groups; the interior is two planes away from every HALO face, so it touches
        no slot an exchange reads or writes)."""
        for _ in range(n):
            if not self.overlap:
                for sim in self.blocks:
                    sim.step(1)
                self._exchange(capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN)
                continue
            for sim, (interior, _) in zip(self.blocks, self.groups):
                if interior is not None:
                    sim.step_box(*interior)
            if self._pending is not None:
                self.main.wait_event(self._pending)
                self._pending = None
            for sim, (_, boundary) in zip(self.blocks, self.groups):
                for lo, hi in boundary:
                    sim.step_box(lo, hi)
            phase = capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN
            self.side.wait_stream(self.main)
            for sim in self.blocks:
                sim.set_stream(self.side)
            try:
                self._exchange(phase)
            finally:
                for sim in self.blocks:
                    sim.set_stream(self.main)
            self._pending = self.side.record_event()
        if self._pending is not None:
            self.main.wait_event(self._pending)
            self._pending = None

    def set_populations(self, f, g=None):
        """Resume from whole-domain logical populations (Q, nz, ny, nx) as populations()
        returns them, from any decomposition or none: each block takes its cells, its ghost
        cells included."""
        f, g = _as_tensor(f), _as_tensor(g)
        for sim, c in zip(self.blocks, self.coords):
            sim.set_populations(part_of(f, c).to(sim.device),
                                None if g is None else part_of(g, c).to(sim.device))

    def _gather(self, parts, lead=0):
        import torch
        dev = self.blocks[0].device
        out = None
        for t, sides, coords in zip(parts, self.sides, self.coords):
            own = t[owned_slices(sides, coords, lead)].to(dev)
            if out is None:
                out = torch.empty(tuple(t.shape[:lead]) + self.w.grid, dtype=t.dtype,
                                  device=dev)
            lo = []
            for a in (2, 1, 0):
                first = coords[a][1 if sides[a][0] else 0]
                lo.append(slice(first, first + own.shape[lead + 2 - a]))
            out[(slice(None),) * lead + tuple(lo)] = own
        return out

    def populations(self):
        """Logical populations of the whole domain, (Q, nz, ny, nx), ghost planes dropped."""
        pops = [sim.populations() for sim in self.blocks]
        f = self._gather([p[0] for p in pops], 1)
        g = self._gather([p[1] for p in pops], 1) if pops[0][1] is not None else None
        return f, g

    def macroscopic(self):
        """rho, u, T of the whole domain (T is None without a thermal lattice)."""
        fields = [sim.macroscopic() for sim in self.blocks]
        rho = self._gather([m[0] for m in fields])
        u = self._gather([m[1] for m in fields], 1)
        T = self._gather([m[2] for m in fields]) if fields[0][2] is not None else None
        return rho, u, T

    def diagnostics(self) -> dict:
        """Whole-domain diagnostics: the blocks' sums (each block leaves its ghost cells out)
        and the Nusselt numbers from them (combine_diagnostics)."""
        vs = [diag_vector(sim.diagnostics(allow_nonfinite=True)) for sim in self.blocks]
        return combine_diagnostics(self.w, [float(x) for x in np.sum(vs, axis=0)])

    def halo_launches_per_step(self) -> int:
        if self.swap:
            return sum((len(self.pairs(a)) + 31) // 32 for a in exchange_axes(self.dim, self.nb))
        return 4 * sum(len(self.pairs(a)) for a in exchange_axes(self.dim, self.nb))

    def halo_bytes_per_step(self) -> float:
        """Bytes the exchanges move between blocks per time step (both ways, every face)."""
        return float(sum(2 * self.face_floats[lo][a] * 4
                         for a in exchange_axes(self.dim, self.nb) for lo, _ in self.pairs(a)))

    def close(self):
        for sim in self.blocks:
            sim.close()


class DistBlockDomain:
    """Block ``rank`` of ``w`` cut into nb = (bx, by, bz) blocks, one per torch.distributed
    rank (world = bx * by * bz).  Each step is followed by the exchange of every split axis,
    z then y then x: per axis the packs, the messages to the two neighbours along that axis
    (halo_messages), and the unpacks, before the next axis packs.  ``transport`` as for
    DistSlabDomain: "device" buffers handed to the process group on the exchange stream
    (NCCL; the host never waits), or "host" page-locked buffers (gloo), where the host waits
    for each axis's packs before sending.  ``overlap``: each step runs as the interior box,
    the wait for the previous exchange, the boundary boxes (block_groups), then the exchange
    on the exchange stream beside the next step's interior."""

    def __init__(self, w, nb, rank: int, world: int, device=None, group=None,
                 transport: str = "device", overlap: bool = False):
        import torch
        nb = tuple(int(v) for v in nb)
        if nb[0] * nb[1] * nb[2] != world:
            raise ValueError("the block counts must multiply to the world size")
        if transport not in ("device", "host"):
            raise ValueError("transport must be 'device' or 'host'")
        self.w, self.nb, self.rank, self.world, self.group = w, nb, rank, world, group
        self.transport, self.overlap = transport, bool(overlap)
        self.periodic = [w.face_flow[2 * a] == "periodic" for a in range(3)]
        self.local, self.sides, self.coords = block_part(w, nb, rank)
        dev = torch.device(device if device is not None else "cuda")
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev)
        self.sim = Simulation(self.local, device=dev, stream=self.main)
        self.interior, self.boundary = block_groups([len(c) for c in self.coords], self.sides,
                                                    w.dim)
        self.axes = exchange_axes(w.dim, nb)
        self.nbs = block_neighbours(rank, nb, self.periodic)
        self.send, self.recv = [], []
        for a in range(3):
            if a in self.axes:
                nfloat = capi.lbm_halo_axis_bytes(self.sim.ctx, a) // 4
                if transport == "host":
                    new = lambda: torch.empty(nfloat, dtype=torch.float32).pin_memory()
                else:
                    new = lambda: torch.empty(nfloat, dtype=torch.float32, device=dev)
                self.send.append([new(), new()])
                self.recv.append([new(), new()])
            else:
                self.send.append(None)
                self.recv.append(None)
        self._packed = None     # host transport: (event after axis k's packs, k, phase)
        self._pending = None    # event: the last exchange's unpacks are queued before it

    @property
    def parity(self) -> int:
        return self.sim.parity

    def init_equilibrium(self):
        import torch
        dev = lambda a: None if a is None else torch.from_numpy(a).to(self.sim.device)
        self.sim.init_equilibrium(dev(self.local.rho0), dev(self.local.u0),
                                  dev(self.local.T_init))

    def _pack_axis(self, k: int, phase: int):
        a = self.axes[k]
        for side in (0, 1):
            if self.nbs[a][side] is not None:
                capi.lbm_halo_axis_pack(self.sim.ctx, a, side, phase, self.send[a][side])

    def _unpack_axis(self, k: int, phase: int, arrived):
        for side, buf in arrived:
            capi.lbm_halo_axis_unpack(self.sim.ctx, self.axes[k], side, phase, buf)

    def _start_exchange(self):
        """Queue this step's exchange on the exchange stream behind the step's last launch:
        with device buffers all of it; with host buffers the first axis's packs."""
        import torch
        if not self.axes:
            return
        phase = capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN
        self.side.wait_stream(self.main)
        self.sim.set_stream(self.side)
        try:
            if self.transport == "host":
                self._pack_axis(0, phase)
                self._packed = (self.side.record_event(), 0, phase)
                return
            with torch.cuda.stream(self.side):
                for k, a in enumerate(self.axes):
                    self._pack_axis(k, phase)
                    arrived = halo_messages(self.nbs[a], self.send[a], self.recv[a], self.group)
                    self._unpack_axis(k, phase, arrived)
        finally:
            self.sim.set_stream(self.main)
        self._pending = self.side.record_event()

    def _finish_exchange(self):
        """Complete the exchange in flight (host transport: per axis, wait for its packs, move
        the messages, queue the unpacks and the next axis's packs) and order it before later
        work on the main stream."""
        if self._packed is not None:
            event, k, phase = self._packed
            self._packed = None
            self.sim.set_stream(self.side)
            try:
                while True:
                    event.synchronize()
                    a = self.axes[k]
                    arrived = halo_messages(self.nbs[a], self.send[a], self.recv[a], self.group)
                    self._unpack_axis(k, phase, arrived)
                    k += 1
                    if k == len(self.axes):
                        break
                    self._pack_axis(k, phase)
                    event = self.side.record_event()
            finally:
                self.sim.set_stream(self.main)
            self._pending = self.side.record_event()
        if self._pending is not None:
            self.main.wait_event(self._pending)
            self._pending = None

    def step(self, n: int = 1):
        """n time steps with their exchanges; returns with the last exchange done (its
        unpacks ordered before later work on the main stream)."""
        for _ in range(n):
            if self.overlap:
                if self.interior is not None:
                    self.sim.step_box(*self.interior)
                self._finish_exchange()
                for lo, hi in self.boundary:
                    self.sim.step_box(lo, hi)
            else:
                self._finish_exchange()
                self.sim.step(1)
            self._start_exchange()
        self._finish_exchange()

    def set_populations(self, f, g=None):
        """Resume this rank's block from whole-domain logical populations (Q, nz, ny, nx)."""
        f, g = _as_tensor(f), _as_tensor(g)
        self.sim.set_populations(part_of(f, self.coords).to(self.sim.device),
                                 None if g is None else part_of(g, self.coords).to(self.sim.device))

    def owned(self, t, lead=0):
        """The owned cells of a local field (ghost planes dropped)."""
        return t[owned_slices(self.sides, self.coords, lead)]

    def populations(self):
        f, g = self.sim.populations()
        return self.owned(f, 1), (None if g is None else self.owned(g, 1))

    def macroscopic(self):
        rho, u, T = self.sim.macroscopic()
        return self.owned(rho), self.owned(u, 1), (None if T is None else self.owned(T))

    def diagnostics(self) -> dict:
        """This rank's own diagnostics (its owned cells)."""
        return self.sim.diagnostics(allow_nonfinite=True)

    def global_diagnostics(self) -> dict:
        """The whole domain's diagnostics: an all-reduce over the ranks (a collective: every
        rank calls it), on the device for the device transport, on the CPU for the host one."""
        dev = self.sim.device if self.transport == "device" else None
        return allreduce_diagnostics(self.w, self.diagnostics(), self.group, dev)

    def close(self):
        self.sim.close()
