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


class SlabDomain:
    """The workload ``w`` split into ``nslabs`` slabs along its outer axis, slab r on
    ``devices[r % len(devices)]``.  The outer axis must be periodic (the slabs form a ring)
    or have WALL faces (the end slabs keep them)."""

    def __init__(self, w, nslabs: int, devices=None):
        import torch
        if getattr(w, "ib_x", None) is not None and len(w.ib_x):
            raise ValueError("slabs do not take immersed-boundary samples")
        self.w = w
        self.dim = w.dim
        self.axis = self.dim - 1                  # outer axis in (x, y, z)
        self.np_axis = 0 if self.dim == 3 else 1  # its axis in a (nz, ny, nx) field
        self.n_outer = w.shape[self.axis]
        lo_face, hi_face = w.face_flow[2 * self.axis], w.face_flow[2 * self.axis + 1]
        self.periodic = lo_face == "periodic"
        if not 1 <= nslabs <= self.n_outer:
            raise ValueError("nslabs must lie in [1, outer extent]")
        devices = list(devices) if devices else [torch.device("cuda")]
        self.ranges = split_ranges(self.n_outer, nslabs)
        self.slabs, self.sides, self.plane_lists, self.buffers = [], [], [], []
        for r, (lo, hi) in enumerate(self.ranges):
            low = self.periodic or r > 0          # ghost plane below the owned ones
            high = self.periodic or r < nslabs - 1
            planes = ([(lo - 1) % self.n_outer] if low else []) + list(range(lo, hi)) + \
                     ([hi % self.n_outer] if high else [])
            faces = list(w.face_flow)
            faces[2 * self.axis] = "halo" if low else lo_face
            faces[2 * self.axis + 1] = "halo" if high else hi_face
            shape = list(w.shape)
            shape[self.axis] = len(planes)
            local = dataclasses.replace(
                w, shape=tuple(shape), face_flow=tuple(faces),
                solid=self._take(w.solid, planes), rho0=self._take(w.rho0, planes),
                u0=self._take(w.u0, planes, 1), T_init=self._take(w.T_init, planes))
            sim = Simulation(local, device=devices[r % len(devices)])
            nfloat = capi.lbm_halo_bytes(sim.ctx) // 4
            self.slabs.append(sim)
            self.sides.append((low, high))
            self.plane_lists.append(planes)
            self.buffers.append([torch.empty(nfloat, dtype=torch.float32, device=sim.device)
                                 for _ in range(2)])   # [low side, high side]
        self.multi_device = len({s.device for s in self.slabs}) > 1

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
        """n time steps, each followed by its exchange (FILL after even, DRAIN after odd)."""
        for _ in range(n):
            for sim in self.slabs:
                sim.step(1)
            self._exchange(capi.LBM_HALO_FILL if self.parity == 1 else capi.LBM_HALO_DRAIN)

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
        """Sums over the slabs (each slab leaves its ghost planes out)."""
        ds = [sim.diagnostics(allow_nonfinite=True) for sim in self.slabs]
        total = lambda key: [float(v) for v in np.sum([d[key] for d in ds], axis=0)]
        return {"mass": sum(d["mass"] for d in ds), "momentum": total("momentum"),
                "force": total("force"), "heat": total("heat"),
                "fluid_cells": sum(d["fluid_cells"] for d in ds),
                "finite": all(d["finite"] for d in ds)}

    def halo_bytes_per_step(self) -> float:
        """Bytes the exchanges move between slabs per time step, averaged over a step pair
        (one FILL and one DRAIN per pair; two buffers per slab face, one each way)."""
        per_face = sum(self.buffers[a][1].numel() * 4 for a, _ in self.pairs())
        return 2 * per_face

    def close(self):
        for sim in self.slabs:
            sim.close()
