"""GB300-native (sm_103a) lattice-Boltzmann collide-and-stream step.

The compute lives in ``liblbm_gb300.so`` (CUDA, C ABI declared in ``include/lbm.h``):
D3Q19 / D2Q9 populations with BGK or MRT collision and D3Q27 populations with
central-moment MRT, Guo forcing with Boussinesq buoyancy, fused D3Q7 / D2Q5 thermal
populations, half-way bounce-back and anti-bounce-back walls through a per-cell link mask,
momentum exchange on solids, an immersed boundary, all streamed in place with the AA
pattern in one fp32 structure-of-arrays buffer (two-buffer layouts for comparison).

* ``capi``      -- one Python function per C entry point (same names).
* ``solver``    -- ``make_config`` and the ``Simulation`` handle.
* ``slabs``     -- a domain split into slabs with the halo exchange (one process, or one
  slab per torch.distributed rank), whole-domain diagnostics and checkpoints.
* ``blocks``    -- a domain cut into blocks along several axes, the same way.
* ``pipeline``  -- independent jobs with host-link copies overlapped with the steps.
* ``workloads`` -- seeded synthetic problems.
"""
from . import capi, workloads  # noqa: F401
from .solver import Simulation, make_config  # noqa: F401

__all__ = ["capi", "workloads", "Simulation", "make_config", "build"]


def build(force: bool = False) -> str:
    """Compile liblbm_gb300.so (sm_103a) in-tree and return its path."""
    from . import _build
    return _build.build(force=force)
