"""Independent jobs on one device state with the host-link copies hidden behind the steps.

A job is: fields from page-locked host memory -> lbm_init_equilibrium -> n steps ->
lbm_macroscopic into page-locked host memory -> lbm_diagnostics.  Run one after another,
each job waits for its host-to-device copy before its first step and for its
device-to-host copy after its last.  Here the uploads run on a copy stream of their own
into double-buffered device staging fields, so job k+1's inputs travel while job k steps.
Events order each staging buffer against the compute stream; nothing is shared between
jobs except the population state, which every job re-initialises.

A copy in flight holds back the kernels issued after it on the other streams: one 2 GB
upload of a 512^3 job held the next steps back for most of its duration, and where it
landed among those launches depended on how far the host had got.  So the uploads are cut
into pieces of about ``piece_bytes`` (at most one piece per step), the steps into as many
groups, and piece i is issued right after group i's launch: a piece (about 43 MB at 512^3
and 50 steps) completes well inside the step it runs beside.  Measured on GB300 at 512^3,
the steps with the next job's upload beside them ran at the rate of the steps alone.
Small jobs take one piece and one group, so their steps keep the library's captured-graph
replay.

Read-outs overlapped the same way (``overlap_readout=True``, through device staging
fields and the copy engine) made the steps beside them slower by more than the copy's own
duration, by an amount that changed from run to run (from no loss to 20 %), and the same
2.15 GB copy engine read-out took 11 ms in one job and 60-74 ms in the next.  So by default
a job's read-out is lbm_macroscopic writing the caller's page-locked host fields itself
(the library resolves them to device-visible addresses), between the job's last step and
the next job's init: a kernel bound by the host link, about 10 ms at 512^3, the same in
every run.  The next job's upload still travels beside the steps.
"""
from __future__ import annotations


def check_jobs(jobs, grid, dim: int, thermal: bool):
    """Raise ValueError unless every job is ((rho, u, T), outputs) with rho and T of shape
    ``grid``, u of shape (dim,) + grid, T present exactly when the lattice is thermal, and
    outputs None or a triple of the same shapes (None entries skip that field)."""
    grid = tuple(grid)
    shapes = (grid, (dim,) + grid, grid)
    names = ("rho", "u", "T")
    for k, job in enumerate(jobs):
        if not isinstance(job, (tuple, list)) or len(job) != 2:
            raise ValueError(f"job {k}: expected (inputs, outputs)")
        ins, outs = job
        if not isinstance(ins, (tuple, list)) or len(ins) != 3:
            raise ValueError(f"job {k}: inputs must be (rho, u, T or None)")
        for i, (t, shape, name) in enumerate(zip(ins, shapes, names)):
            needed = i < 2 or thermal
            if t is None:
                if needed:
                    raise ValueError(f"job {k}: input {name} is required")
                continue
            if not needed:
                raise ValueError(f"job {k}: input {name} given for a lattice without it")
            if tuple(t.shape) != shape:
                raise ValueError(f"job {k}: input {name} has shape {tuple(t.shape)}, "
                                 f"expected {shape}")
        if outs is None:
            continue
        if not isinstance(outs, (tuple, list)) or len(outs) != 3:
            raise ValueError(f"job {k}: outputs must be None or (rho, u, T or None)")
        for t, shape, name in zip(outs, shapes, names):
            if t is not None and tuple(t.shape) != shape:
                raise ValueError(f"job {k}: output {name} has shape {tuple(t.shape)}, "
                                 f"expected {shape}")


def _pieces(n: int, parts: int):
    """[lo, hi) ranges cutting range(n) into ``parts`` nearly equal pieces."""
    return [(n * i // parts, n * (i + 1) // parts) for i in range(parts)]


class JobPipeline:
    """Runs jobs on ``sim`` (moved onto a compute stream of its own) with overlapped
    host-link copies.  Every host tensor must be page-locked and contiguous."""

    def __init__(self, sim, piece_bytes: int = 32 << 20, overlap_readout: bool = False):
        import torch
        self.sim = sim
        self.piece_bytes = int(piece_bytes)
        self.overlap_readout = bool(overlap_readout)
        dev = sim.device
        grid, dim, thermal = sim.grid, sim.dim, bool(sim.QT)

        def fields():
            return [torch.empty(grid, dtype=torch.float32, device=dev),
                    torch.empty((dim,) + grid, dtype=torch.float32, device=dev),
                    torch.empty(grid, dtype=torch.float32, device=dev) if thermal else None]

        self.inp = [fields(), fields()]
        self.out = [fields(), fields()] if self.overlap_readout else None
        self.compute = torch.cuda.Stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        sim.set_stream(self.compute.cuda_stream)

    @staticmethod
    def _copy_piece(pairs, i: int, parts: int):
        """Piece i of ``parts`` of every (destination, source) pair, flattened."""
        for dst, src in pairs:
            if dst is None or src is None:
                continue
            d, s = dst.view(-1), src.view(-1)
            lo, hi = _pieces(d.numel(), parts)[i]
            if hi > lo:
                d[lo:hi].copy_(s[lo:hi], non_blocking=True)

    def run(self, jobs, steps: int):
        """jobs: sequence of (inputs, outputs); inputs = (rho, u, T or None), outputs =
        (rho, u, T or None) or None to skip the read-out, all page-locked host tensors.
        Returns each job's diagnostics (dict, as Simulation.diagnostics)."""
        import torch
        jobs = list(jobs)
        check_jobs(jobs, self.sim.grid, self.sim.dim, bool(self.sim.QT))
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        staged, staging_free, written, drained = ev(), ev(), ev(), ev()
        # another pipeline built on the same simulation since may have moved it
        self.sim.set_stream(self.compute.cuda_stream)
        # the compute stream starts after whatever the caller queued before
        self.compute.wait_stream(torch.cuda.current_stream(self.sim.device))
        field_bytes = sum(t.numel() * t.element_size() for t in self.inp[0] if t is not None)
        parts = max(1, min(steps, field_bytes // max(1, self.piece_bytes)))
        groups = _pieces(steps, parts)

        def upload_pairs(k):
            return list(zip(self.inp[k % 2], jobs[k][0]))

        def readout_pairs(k, outs):
            return list(zip(outs, self.out[k % 2]))

        diags = []
        if jobs:                       # the first job's inputs in one piece
            with torch.cuda.stream(self.h2d):
                self._copy_piece(upload_pairs(0), 0, 1)
                staged[0].record(self.h2d)
        pending = None                 # (job, outputs) whose read-out travels during this job,
                                       # with overlap_readout
        for k, (_, outs) in enumerate(jobs):
            s = k % 2
            up = k + 1 < len(jobs)
            if up and k + 1 >= 2:      # job k + 1's staging buffer held job k - 1's inputs
                self.h2d.wait_event(staging_free[(k + 1) % 2])
            if pending is not None:
                self.d2h.wait_event(written[pending[0] % 2])
            self.compute.wait_event(staged[s])
            self.sim.init_equilibrium(*self.inp[s])
            staging_free[s].record(self.compute)
            for i, (a, b) in enumerate(groups):
                if b > a:
                    self.sim.step(b - a)
                if up:
                    with torch.cuda.stream(self.h2d):
                        self._copy_piece(upload_pairs(k + 1), i, parts)
                if pending is not None:
                    with torch.cuda.stream(self.d2h):
                        self._copy_piece(readout_pairs(*pending), i, parts)
            if up:
                staged[(k + 1) % 2].record(self.h2d)
            if pending is not None:
                drained[pending[0] % 2].record(self.d2h)
                pending = None
            if outs is not None and self.overlap_readout:
                self.compute.wait_event(drained[s])     # the read-out of job k - 2
                self.sim.macroscopic(*self.out[s])
                written[s].record(self.compute)
                pending = (k, outs)
            elif outs is not None:     # the read-out kernel writes the host fields itself
                self.sim.macroscopic(*outs)
            diags.append(self.sim.diagnostics(allow_nonfinite=True))
        if pending is not None:        # the last job's read-out in one piece
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(written[pending[0] % 2])
                self._copy_piece(readout_pairs(*pending), 0, 1)
                drained[pending[0] % 2].record(self.d2h)
        self.d2h.synchronize()
        self.compute.synchronize()
        return diags
