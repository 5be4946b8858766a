"""Independent jobs on one device state with the host-link copies hidden behind the steps.

A job is: fields from page-locked host memory -> lbm_init_equilibrium -> n steps ->
lbm_macroscopic into page-locked host memory -> lbm_diagnostics.  Run one after another,
each job waits for its host-to-device copy before its first step and for its
device-to-host copy after its last.  Here the copies run on two copy streams of their own
(the host link is full duplex) into and out of double-buffered device staging fields:
job k+1's inputs travel while job k steps, and job k's outputs travel while job k+1 steps.
Events order each staging buffer against the compute stream; nothing is shared between
jobs except the population state, which every job re-initialises.

A device-to-host copy into page-locked host memory holds back the kernels issued after it
on the other streams until it completes.  On GB300, the next job's init waited for the
whole 12.6 ms read-out of a 512^3 job, so the pipeline ran slower than the serial path.
So job k's read-out is issued only after job k+1's init, steps and read-out kernel are
queued, and it runs beside job k+1's steps.
"""
from __future__ import annotations


class JobPipeline:
    """Runs jobs on ``sim`` (moved onto a compute stream of its own) with overlapped
    host-link copies.  Every host tensor must be page-locked and contiguous."""

    def __init__(self, sim):
        import torch
        self.sim = sim
        dev = sim.device
        grid, dim, thermal = sim.grid, sim.dim, bool(sim.QT)

        def fields():
            return [torch.empty(grid, dtype=torch.float32, device=dev),
                    torch.empty((dim,) + grid, dtype=torch.float32, device=dev),
                    torch.empty(grid, dtype=torch.float32, device=dev) if thermal else None]

        self.inp = [fields(), fields()]
        self.out = [fields(), fields()]
        self.compute = torch.cuda.Stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        sim.set_stream(self.compute.cuda_stream)

    def run(self, jobs, steps: int):
        """jobs: sequence of (inputs, outputs); inputs = (rho, u, T or None), outputs =
        (rho, u, T or None) or None to skip the read-out, all page-locked host tensors.
        Returns each job's diagnostics (dict, as Simulation.diagnostics)."""
        import torch
        jobs = list(jobs)
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        staged, staging_free, written, drained = ev(), ev(), ev(), ev()
        # the compute stream starts after whatever the caller queued before
        self.compute.wait_stream(torch.cuda.current_stream(self.sim.device))

        def upload(k):
            s = k % 2
            with torch.cuda.stream(self.h2d):
                if k >= 2:
                    self.h2d.wait_event(staging_free[s])
                for dst, src in zip(self.inp[s], jobs[k][0]):
                    if src is not None:
                        dst.copy_(src, non_blocking=True)
                staged[s].record(self.h2d)

        def readout(k, outs):
            s = k % 2
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(written[s])
                for dst, src in zip(outs, self.out[s]):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
                drained[s].record(self.d2h)

        diags = []
        pending = None                  # (job, outputs) whose read-out waits for the next job
        if jobs:
            upload(0)
        for k, (_, outs) in enumerate(jobs):
            s = k % 2
            if k + 1 < len(jobs):
                upload(k + 1)
            self.compute.wait_event(staged[s])
            self.sim.init_equilibrium(*self.inp[s])
            staging_free[s].record(self.compute)
            self.sim.step(steps)
            if outs is not None:
                self.compute.wait_event(drained[s])     # the read-out of job k - 2
                self.sim.macroscopic(*self.out[s])
                written[s].record(self.compute)
            if pending is not None:                     # job k - 1's read-out, behind job k
                readout(*pending)
                pending = None
            diags.append(self.sim.diagnostics(allow_nonfinite=True))
            if outs is not None:
                pending = (k, outs)
        if pending is not None:
            readout(*pending)
        self.d2h.synchronize()
        return diags
