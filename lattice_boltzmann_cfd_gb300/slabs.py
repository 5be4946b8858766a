"""A domain split into slabs along its outer axis (z in 3-D, y in 2-D): one library context
per slab, with the direction-selective halo exchange driven from the host.

This is the mono-dimensional partitioning of "Multi-GPU thermal lattice Boltzmann
simulations using OpenACC and MPI" (Sec. 3): each slab holds one ghost plane per inner
face, and only the populations that cross a face travel, as contiguous buffers.  On top of
the in-place AA pattern only odd steps read or write across a slab face, which gives one
exchange after every step:
  after an even step, FILL: a neighbour's boundary plane -> my ghost plane (the slots that
    my boundary cells read during the odd step, and from which the logical state of those
    cells is read while the parity is 1);
  after an odd step, DRAIN: my ghost plane -> the neighbour's boundary plane (the slots my
    boundary cells wrote into the ghost plane).
Each move is a pack kernel into a buffer, a buffer copy when the slabs sit on different
devices, and an unpack kernel, all in stream order; no kernel waits for another.  Between
steps, the state of every owned cell is therefore what a single domain would hold, bit for
bit.

Two drivers share the slicing: SlabDomain holds every slab in one process (on one device or
several); DistSlabDomain is one slab per torch.distributed rank, its buffers moved by
point-to-point messages (ring_exchange).  The block partitioning of blocks.py shares this
module's helpers: the split of a field into a part's planes (part_of), the whole-domain
diagnostics of the parts (combine_diagnostics, allreduce_diagnostics) and the point-to-point
messages (halo_messages).

Overlap ("Multi-GPU thermal lattice Boltzmann simulations using OpenACC and MPI", Sec. 4:
the boundary layers first, then the exchange beside the interior update).  With
``overlap=True`` each step runs through lbm_step_planes as: the interior planes; a wait for
the previous step's exchange; the boundary planes (the ghost plane and the first owned
plane at each HALO face); then this step's exchange on a second stream, where it runs beside
the next step's interior planes.  A pack reads only slots the interior update leaves alone,
and an unpack writes only slots that the boundary planes' next step reads first, so the
result is bit for bit that of the plain order.  The host never waits for the device, except
where the messages themselves go through the host (page-locked buffers over a CPU back-end
such as gloo): there the host waits for the pack alone, after the next interior launch is
queued.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import capi
from .solver import Simulation


def split_ranges(n: int, parts: int):
    """Contiguous, nearly equal [lo, hi) ranges covering range(n)."""
    edges = [round(i * n / parts) for i in range(parts + 1)]
    return [(edges[i], edges[i + 1]) for i in range(parts)]


def outer_axis(w):
    """(axis in (x, y, z), axis in a (nz, ny, nx) field) of the slab direction."""
    return w.dim - 1, (0 if w.dim == 3 else 1)


# ------------------------------------------------------------------ checkpoint / resume ---

def part_of(t, coords, lead=1):
    """The part of a whole-domain field t (``lead`` leading axes, then z, y, x) at the domain
    coordinates coords = (x list, y list, z list) of a part's local planes (ghost planes
    included), as a contiguous tensor on t's device."""
    import torch
    for a, dim in ((2, lead), (1, lead + 1), (0, lead + 2)):
        idx = torch.as_tensor(coords[a], dtype=torch.long, device=t.device)
        t = torch.index_select(t, dim, idx)
    return t.contiguous()


def _device_index(d) -> int:
    """The CUDA device index of a device or device name ("cuda" = the current device)."""
    import torch
    d = torch.device(d)
    return d.index if d.index is not None else torch.cuda.current_device()


def _as_tensor(a):
    import torch
    return a if a is None or isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))


# ------------------------------------------------------------- whole-domain diagnostics ---

# The extensive sums of lbm_diagnostics, in the order diag_vector packs them.
_DIAG_SUMS = (("mass", 1), ("momentum", 3), ("force", 3), ("heat", 6), ("uT", 3),
              ("fluid_cells", 1))


def diag_vector(d: dict):
    """The extensive sums of one part's diagnostics as a flat list, then 0 / 1 for finite /
    not finite (so that a sum over parts counts the parts that are not)."""
    v = []
    for key, n in _DIAG_SUMS:
        v += [float(x) for x in (d[key] if n > 1 else [d[key]])]
    return v + [0.0 if d["finite"] else 1.0]


def combine_diagnostics(w, v) -> dict:
    """Whole-domain diagnostics of workload ``w`` from the summed diag_vector of its parts
    (slabs or blocks, each of which leaves its ghost cells out): the sums, and the Nusselt
    numbers recomputed from them with the whole domain's extents, as lbm_diagnostics does for
    one domain (wall heat |heat| H / (dT A) of the hottest and coldest DIRICHLET faces, and
    the volume average 1 + <u_a T> H / (kappa dT) along their axis)."""
    from .solver import make_config
    out, i = {}, 0
    for key, n in _DIAG_SUMS:
        out[key] = list(v[i:i + n]) if n > 1 else v[i]
        i += n
    out["fluid_cells"] = int(round(out["fluid_cells"]))
    out["finite"] = v[i] == 0.0
    out["nu_hot"] = out["nu_cold"] = out["nu_volume"] = 0.0
    cfg, _ = make_config(w)
    dirichlet = [f for f in range(2 * w.dim)
                 if cfg.thermal and cfg.face_flow[f] == capi.LBM_FACE_WALL
                 and cfg.face_T[f] == capi.LBM_TFACE_DIRICHLET]
    if not dirichlet:
        return out
    hot = max(dirichlet, key=lambda f: (cfg.T_wall[f], -f))    # the first of equal faces
    cold = min(dirichlet, key=lambda f: (cfg.T_wall[f], f))
    dT = cfg.T_wall[hot] - cfg.T_wall[cold]
    if dT <= 0:
        return out
    n = list(w.shape)
    cells = n[0] * n[1] * n[2]
    nusselt = lambda f: abs(out["heat"][f]) * n[f // 2] / (dT * cells / n[f // 2])
    out["nu_hot"], out["nu_cold"] = nusselt(hot), nusselt(cold)
    a = hot // 2
    if cold // 2 == a and out["fluid_cells"] > 0:
        omega = (4.0 + cfg.a_T) / 10.0 if cfg.thermal == 5 else (6.0 + cfg.a_T) / 21.0
        kappa = omega * (1.0 / cfg.s_T[1 + a] - 0.5)
        sign = 1.0 if hot % 2 == 0 else -1.0
        out["nu_volume"] = 1.0 + sign * out["uT"][a] / out["fluid_cells"] * n[a] / (kappa * dT)
    return out


def allreduce_diagnostics(w, d: dict, group=None, device=None) -> dict:
    """combine_diagnostics over every rank of a process group: one all-reduce (sum) of the
    ranks' diag_vector, in fp64, on ``device`` (None: the CPU, for gloo)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(diag_vector(d), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return combine_diagnostics(w, t.cpu().tolist())


def slab_part(w, nslabs: int, r: int):
    """Slab r of ``w`` split into ``nslabs`` along its outer axis: (local workload, (low,
    high) ghost flags, the domain plane of each local plane).  A periodic outer axis wraps
    (the slabs form a ring); the end slabs of a walled one keep their faces."""
    axis, np_axis = outer_axis(w)
    n_outer = w.shape[axis]
    lo_face, hi_face = w.face_flow[2 * axis], w.face_flow[2 * axis + 1]
    periodic = lo_face == "periodic"
    if not 1 <= nslabs <= n_outer:
        raise ValueError("nslabs must lie in [1, outer extent]")
    if getattr(w, "ib_x", None) is not None and len(w.ib_x):
        raise ValueError("slabs do not take immersed-boundary samples")
    lo, hi = split_ranges(n_outer, nslabs)[r]
    low = periodic or r > 0
    high = periodic or r < nslabs - 1
    planes = ([(lo - 1) % n_outer] if low else []) + list(range(lo, hi)) + \
             ([hi % n_outer] if high else [])
    faces = list(w.face_flow)
    faces[2 * axis] = "halo" if low else lo_face
    faces[2 * axis + 1] = "halo" if high else hi_face
    shape = list(w.shape)
    shape[axis] = len(planes)

    def take(a, lead=0):
        if a is None:
            return None
        return np.ascontiguousarray(np.take(a, planes, axis=np_axis + lead))

    local = dataclasses.replace(
        w, shape=tuple(shape), face_flow=tuple(faces), solid=take(w.solid),
        rho0=take(w.rho0), u0=take(w.u0, 1), T_init=take(w.T_init))
    return local, (low, high), planes


def plane_groups(n: int, low: bool, high: bool):
    """(interior, boundary) lists of [lo, hi) outer-axis plane ranges of a slab with ``n``
    local planes and ghost planes at the low / high end when ``low`` / ``high``.  The
    boundary ranges are the ghost plane and the first owned plane of each HALO face; the
    interior is what lies between.  A slab too thin for an interior is all boundary."""
    lo_b = 2 if low else 0
    hi_b = n - 2 if high else n
    if hi_b <= lo_b:
        return [], [(0, n)]
    boundary = ([(0, lo_b)] if low else []) + ([(hi_b, n)] if high else [])
    return [(lo_b, hi_b)], boundary


def ring_neighbours(rank: int, world: int, periodic: bool):
    """(low, high) neighbour ranks of slab ``rank`` (None at the end of a walled axis)."""
    lo_nb = rank - 1 if rank > 0 else (world - 1 if periodic else None)
    hi_nb = rank + 1 if rank < world - 1 else (0 if periodic else None)
    return lo_nb, hi_nb


def ring_messages(rank: int, world: int, periodic: bool, send, recv, group=None):
    """Move packed buffers between neighbours; returns [(side, buffer to unpack there)].

    My side-s buffer goes to the neighbour's opposite side.  Messages carry as tag the side
    they land on, and are posted in one fixed order (sends of sides 0, 1; receives of the
    neighbours' side 0, then side 1), so that back-ends which match point-to-point messages
    by order (NCCL) pair them right even when both neighbours are the same rank.  A ring of
    one slab unpacks its own buffers, crossed."""
    nbs = ring_neighbours(rank, world, periodic)
    if world == 1:
        return [(0, send[1]), (1, send[0])] if periodic else []
    return halo_messages(nbs, send, recv, group)


def halo_messages(nbs, send, recv, group=None):
    """Send send[s] to rank nbs[s] and receive recv[s] from it, for each side s whose
    neighbour is not None; returns [(side, buffer to unpack there)].  The messages are
    tagged and posted as ring_messages describes."""
    import torch.distributed as dist
    ops = []
    for side in (0, 1):
        if nbs[side] is not None:
            ops.append(dist.P2POp(dist.isend, send[side], nbs[side], group, tag=1 - side))
    # the neighbour's side-0 buffer lands on my side 1, its side-1 buffer on my side 0
    for their_side in (0, 1):
        mine = 1 - their_side
        if nbs[mine] is not None:
            ops.append(dist.P2POp(dist.irecv, recv[mine], nbs[mine], group, tag=mine))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return [(side, recv[side]) for side in (0, 1) if nbs[side] is not None]


def ring_exchange(rank: int, world: int, periodic: bool, phase: int, pack, unpack, send,
                  recv, group=None, sync=None):
    """One halo exchange of slab ``rank`` with its neighbours over torch.distributed.

    pack(side, phase, buf) fills send[side]; unpack(side, phase, buf) consumes a buffer;
    sync(), if given, runs after the packs and again after the receives (to order device
    work around the messages).
    My side-s buffer goes to the neighbour's opposite side.  Messages carry as tag the side
    they land on, and are posted in one fixed order (sends of sides 0, 1; receives of the
    neighbours' side 0, then side 1), so that back-ends which match point-to-point messages
    by order (NCCL) pair them right even when both neighbours are the same rank."""
    nbs = ring_neighbours(rank, world, periodic)
    for side in (0, 1):
        if nbs[side] is not None:
            pack(side, phase, send[side])
    if sync is not None:
        sync()
    arrived = ring_messages(rank, world, periodic, send, recv, group)
    if sync is not None and world > 1:
        sync()
    for side, buf in arrived:
        unpack(side, phase, buf)


class SlabDomain:
    """The workload ``w`` split into ``nslabs`` slabs along its outer axis, slab r on
    ``devices[r % len(devices)]``.  The outer axis must be periodic (the slabs form a ring)
    or have WALL faces (the end slabs keep them).

    ``overlap``: run each step as interior planes, then boundary planes, with the exchange
    on a second stream beside the next step's interior (one device only).
    ``exchange``: as for BlockDomain ("auto": the buffer-free swap on one device)."""

    def __init__(self, w, nslabs: int, devices=None, overlap: bool = False,
                 exchange: str = "auto"):
        import torch
        if exchange not in ("auto", "swap", "buffers"):
            raise ValueError("exchange must be 'auto', 'swap' or 'buffers'")
        self.w = w
        self.dim = w.dim
        self.axis, self.np_axis = outer_axis(w)
        self.n_outer = w.shape[self.axis]
        self.periodic = w.face_flow[2 * self.axis] == "periodic"
        devices = list(devices) if devices else [torch.device("cuda")]
        self.multi_device = len({_device_index(d) for d in devices[:nslabs]}) > 1
        if exchange == "swap" and self.multi_device:
            raise ValueError("the buffer-free swap needs every slab on one device")
        self.swap = exchange == "swap" or (exchange == "auto" and not self.multi_device)
        self.slabs, self.sides, self.plane_lists, self.buffers = [], [], [], []
        self.groups, self.face_floats = [], []
        for r in range(nslabs):
            local, sides, planes = slab_part(w, nslabs, r)
            sim = Simulation(local, device=devices[r % len(devices)])
            nfloat = capi.lbm_halo_bytes(sim.ctx) // 4
            self.slabs.append(sim)
            self.sides.append(sides)
            self.plane_lists.append(planes)
            self.groups.append(plane_groups(len(planes), *sides))
            self.face_floats.append(nfloat)
            # [low side, high side]; the swap needs none
            self.buffers.append(None if self.swap else
                                [torch.empty(nfloat, dtype=torch.float32, device=sim.device)
                                 for _ in range(2)])
        self.overlap = bool(overlap)
        if self.overlap and self.multi_device:
            raise ValueError("overlap needs every slab on one device")
        dev = self.slabs[0].device
        # the contexts' stream (torch's current stream at creation) and the exchange stream
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev) if self.overlap else None
        self._pending = None    # event: the last exchange's unpacks are queued before it

    def _take(self, a, planes, lead=0):
        if a is None:
            return None
        return np.ascontiguousarray(np.take(a, planes, axis=self.np_axis + lead))

    # (slab a, high side) faces (slab b, low side); the last pair closes a periodic ring
    def pairs(self):
        n = len(self.slabs)
        pairs = [(r, r + 1) for r in range(n - 1)]
        if self.periodic:
            pairs.append((n - 1, 0))
        return pairs

    def _sync(self):
        import torch
        if self.multi_device:
            for d in {s.device for s in self.slabs}:
                torch.cuda.synchronize(d)

    def _exchange(self, phase: int):
        pairs = self.pairs()
        if self.swap:         # every face in one launch (32 per launch at most)
            for k in range(0, len(pairs), 32):
                chunk = pairs[k:k + 32]
                capi.lbm_halo_axis_swap_many([self.slabs[a].ctx for a, _ in chunk],
                                             [self.slabs[b].ctx for _, b in chunk],
                                             self.axis, phase)
            return
        for a, b in pairs:
            capi.lbm_halo_pack(self.slabs[a].ctx, 1, phase, self.buffers[a][1])
            capi.lbm_halo_pack(self.slabs[b].ctx, 0, phase, self.buffers[b][0])
        self._sync()
        for a, b in pairs:
            to_a = self.buffers[b][0].to(self.slabs[a].device)
            to_b = self.buffers[a][1].to(self.slabs[b].device)
            capi.lbm_halo_unpack(self.slabs[a].ctx, 1, phase, to_a)
            capi.lbm_halo_unpack(self.slabs[b].ctx, 0, phase, to_b)
        self._sync()

    def _exchange_on_side(self, phase: int):
        """This step's exchange on the side stream, after the boundary planes on the main
        stream; leaves an event the next boundary planes wait for."""
        self.side.wait_stream(self.main)
        for sim in self.slabs:
            sim.set_stream(self.side)
        try:
            self._exchange(phase)
        finally:
            for sim in self.slabs:
                sim.set_stream(self.main)
        self._pending = self.side.record_event()

    def _wait_pending(self):
        if self._pending is not None:
            self.main.wait_event(self._pending)
            self._pending = None

    @property
    def parity(self) -> int:
        return self.slabs[0].parity

    def init_equilibrium(self):
        """Every slab from the workload's initial fields (its ghost planes included)."""
        import torch
        for sim, planes in zip(self.slabs, self.plane_lists):
            def dev(a, lead=0):
                t = self._take(a, planes, lead)
                return None if t is None else torch.from_numpy(t).to(sim.device)
            sim.init_equilibrium(dev(self.w.rho0), dev(self.w.u0, 1), dev(self.w.T_init))

    def step(self, n: int = 1):
        """n time steps, each followed by its exchange (FILL after even, DRAIN after odd).
        Returns with every exchange ordered before later work on the main stream."""
        for _ in range(n):
            if not self.overlap:
                for sim in self.slabs:
                    sim.step(1)
                self._exchange(capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN)
                continue
            for sim, (interior, _) in zip(self.slabs, self.groups):
                for lo, hi in interior:
                    sim.step_planes(lo, hi)
            self._wait_pending()
            for sim, (_, boundary) in zip(self.slabs, self.groups):
                for lo, hi in boundary:
                    sim.step_planes(lo, hi)
            self._exchange_on_side(capi.LBM_HALO_FILL if self.parity == 1
                                   else capi.LBM_HALO_DRAIN)
        self._wait_pending()

    def _coords(self, r):
        """(x, y, z) domain coordinates of slab r's local planes."""
        c = [list(range(n)) for n in self.w.shape]
        c[self.axis] = list(self.plane_lists[r])
        return c

    def set_populations(self, f, g=None):
        """Resume from whole-domain logical populations (Q, nz, ny, nx) as populations()
        returns them, from any decomposition or none: each slab takes its planes, its ghost
        planes included, so the exchange state is the one the step after needs at either
        parity."""
        f, g = _as_tensor(f), _as_tensor(g)
        for r, sim in enumerate(self.slabs):
            c = self._coords(r)
            sim.set_populations(part_of(f, c).to(sim.device),
                                None if g is None else part_of(g, c).to(sim.device))

    def _owned(self, t, r, lead=0):
        low, high = self.sides[r]
        idx = [slice(None)] * t.dim()
        idx[self.np_axis + lead] = slice(1 if low else 0, t.shape[self.np_axis + lead] -
                                         (1 if high else 0))
        return t[tuple(idx)]

    def _gather(self, parts, lead=0):
        import torch
        dev = self.slabs[0].device
        owned = [self._owned(t, r, lead).to(dev) for r, t in enumerate(parts)]
        return torch.cat(owned, dim=self.np_axis + lead)

    def populations(self):
        """Logical populations of the whole domain, (Q, nz, ny, nx), ghost planes dropped."""
        pops = [sim.populations() for sim in self.slabs]
        f = self._gather([p[0] for p in pops], 1)
        g = self._gather([p[1] for p in pops], 1) if pops[0][1] is not None else None
        return f, g

    def macroscopic(self):
        """rho, u, T of the whole domain (T is None without a thermal lattice)."""
        fields = [sim.macroscopic() for sim in self.slabs]
        rho = self._gather([m[0] for m in fields])
        u = self._gather([m[1] for m in fields], 1)
        T = self._gather([m[2] for m in fields]) if fields[0][2] is not None else None
        return rho, u, T

    def diagnostics(self) -> dict:
        """Whole-domain diagnostics: the slabs' sums (each slab leaves its ghost planes out)
        and the Nusselt numbers from them (combine_diagnostics)."""
        vs = [diag_vector(sim.diagnostics(allow_nonfinite=True)) for sim in self.slabs]
        return combine_diagnostics(self.w, [float(x) for x in np.sum(vs, axis=0)])

    def halo_bytes_per_step(self) -> float:
        """Bytes the exchanges move between slabs per time step, averaged over a step pair
        (one FILL and one DRAIN per pair; two buffers per slab face, one each way)."""
        per_face = sum(self.face_floats[a] * 4 for a, _ in self.pairs())
        return 2 * per_face

    def close(self):
        for sim in self.slabs:
            sim.close()


class DistSlabDomain:
    """Slab ``rank`` of ``w`` split into ``world`` slabs, one per torch.distributed rank
    (one process per GPU).  Every step is followed by the exchange of its halos with the
    neighbouring ranks (FILL after even, DRAIN after odd steps), so between steps the owned
    planes hold what one undivided domain would hold.

    ``transport``: "device" keeps the halo buffers in device memory and hands them to the
    process group on the exchange stream (a GPU back-end such as NCCL: the exchange is
    ordered by streams and the host does not wait); "host" keeps them in page-locked host
    memory, which the halo kernels write and read directly, for a CPU back-end such as gloo
    (the host waits for the pack before sending).
    ``overlap``: interior planes, boundary planes, then the exchange beside the next step's
    interior (see the module notes); otherwise each step is followed by its exchange."""

    def __init__(self, w, rank: int, world: int, device=None, group=None,
                 transport: str = "device", overlap: bool = False):
        import torch
        if transport not in ("device", "host"):
            raise ValueError("transport must be 'device' or 'host'")
        self.w, self.rank, self.world, self.group = w, rank, world, group
        self.transport, self.overlap = transport, bool(overlap)
        self.axis, self.np_axis = outer_axis(w)
        self.periodic = w.face_flow[2 * self.axis] == "periodic"
        self.range = split_ranges(w.shape[self.axis], world)[rank]
        local, self.sides, self.planes = slab_part(w, world, rank)
        self.local = local
        dev = torch.device(device if device is not None else "cuda")
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev)
        self.sim = Simulation(local, device=dev, stream=self.main)
        self.interior, self.boundary = plane_groups(len(self.planes), *self.sides)
        nfloat = capi.lbm_halo_bytes(self.sim.ctx) // 4
        if transport == "host":
            new = lambda: torch.empty(nfloat, dtype=torch.float32).pin_memory()
        else:
            new = lambda: torch.empty(nfloat, dtype=torch.float32, device=dev)
        self.send = [new(), new()]
        self.recv = [new(), new()]
        self._packed = None     # (event after the packs, phase) awaiting its messages
        self._pending = None    # event: the unpacks of the last exchange are queued before it

    @property
    def parity(self) -> int:
        return self.sim.parity

    def init_equilibrium(self):
        import torch
        dev = lambda a: None if a is None else torch.from_numpy(a).to(self.sim.device)
        self.sim.init_equilibrium(dev(self.local.rho0), dev(self.local.u0),
                                  dev(self.local.T_init))

    def _pack(self, side, phase, buf):
        capi.lbm_halo_pack(self.sim.ctx, side, phase, buf)

    def _unpack(self, side, phase, buf):
        capi.lbm_halo_unpack(self.sim.ctx, side, phase, buf)

    def _start_exchange(self):
        """Queue this step's packs on the exchange stream behind the step's last planes;
        with device buffers, the messages and the unpacks too."""
        import torch
        phase = capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN
        nbs = ring_neighbours(self.rank, self.world, self.periodic)
        self.side.wait_stream(self.main)
        self.sim.set_stream(self.side)
        try:
            for side in (0, 1):
                if nbs[side] is not None:
                    self._pack(side, phase, self.send[side])
            if self.transport == "host":
                self._packed = (self.side.record_event(), phase)
                return
            with torch.cuda.stream(self.side):
                arrived = ring_messages(self.rank, self.world, self.periodic, self.send,
                                        self.recv, self.group)
            for side, buf in arrived:
                self._unpack(side, phase, buf)
        finally:
            self.sim.set_stream(self.main)
        self._pending = self.side.record_event()

    def _finish_exchange(self):
        """Complete the exchange in flight (host transport: wait for the packs, move the
        messages, queue the unpacks) and order it before later work on the main stream."""
        if self._packed is not None:
            event, phase = self._packed
            self._packed = None
            event.synchronize()
            arrived = ring_messages(self.rank, self.world, self.periodic, self.send,
                                    self.recv, self.group)
            self.sim.set_stream(self.side)
            try:
                for side, buf in arrived:
                    self._unpack(side, phase, buf)
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
                for lo, hi in self.interior:
                    self.sim.step_planes(lo, hi)
                self._finish_exchange()
                for lo, hi in self.boundary:
                    self.sim.step_planes(lo, hi)
            else:
                self._finish_exchange()
                self.sim.step(1)
            self._start_exchange()
        self._finish_exchange()

    def set_populations(self, f, g=None):
        """Resume this rank's slab from whole-domain logical populations (Q, nz, ny, nx)."""
        c = [list(range(n)) for n in self.w.shape]
        c[self.axis] = list(self.planes)
        f, g = _as_tensor(f), _as_tensor(g)
        self.sim.set_populations(part_of(f, c).to(self.sim.device),
                                 None if g is None else part_of(g, c).to(self.sim.device))

    def owned(self, t, lead=0):
        """The owned planes of a local field (ghost planes dropped)."""
        low, high = self.sides
        idx = [slice(None)] * t.dim()
        ax = self.np_axis + lead
        idx[ax] = slice(1 if low else 0, t.shape[ax] - (1 if high else 0))
        return t[tuple(idx)]

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
