"""Throughput of the fused lattice-Boltzmann step on GB300, in MLUPS.

One benchmark step is one submission of the hot path: ``--lbm-steps`` time steps of the
fused AA collide-and-stream kernel (alternating even and odd forms) followed by the
diagnostics reduction (mass, momentum, solid force, wall heat flux) read back to the
host.  MLUPS = cells x time steps / seconds / 1e6, counting every lattice cell (the
MLUPS metric of the multi-GPU thermal LBM page; "cell updates per second" of the
streaming-layout page).

Legs, all printed on one JSON line by rank 0:
  value         device-resident state, K timed steps between CUDA events (max over ranks)
  roofline      the step kernel's achieved algorithmic bandwidth (bytes per cell update
                x cells / average launch time) against the measured HBM copy bandwidth
  e2e           the same metric through the C ABI with page-locked HOST fields: each
                step uploads rho, u (T), initialises, steps, and writes rho, u (T) back
  cpu_baseline  the fp64 oracle on the host cores on a bounded sample of the workload
  secondary     the other workloads of the target (thermal cavities, 128^3) briefly

``--impl reference`` times the oracle instead (the reference arm: a slow, plain CPU
program on this machine's host cores), one bounded sample step per benchmark step.
Multi-GPU runs (torchrun) are independent replicas, one per GPU ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLUPS at 1 GB300 (D3Q19 MRT fp32, AA) and % of HBM bandwidth roofline"
UNIT = "MLUPS"

# Algorithmic bytes per cell update: populations read once and written once, fp32.
BYTES_PER_CELL = {(19, 0): 152, (19, 7): 208, (9, 0): 72, (9, 5): 112, (27, 0): 216}

# DRAM bytes per cell update of the step kernel measured with ncu (dram__bytes_read.sum +
# dram__bytes_write.sum per launch / cells), with a hash of the kernel sources they were
# taken on; reported as "traffic" only while the sources are unchanged.
NCU_TRAFFIC = {
    # ncu --set full, one even + one odd launch at 256^3 (see profiles/), scaled by cells
    "d3q19_mrt_periodic_512": {"bytes_per_cell": 148.66, "src_hash": "a54b079d3d377279"},
    "cavity3d_512": {"bytes_per_cell": 204.77, "src_hash": "a54b079d3d377279"},
}


# The files that define the step kernels (device code and its instantiations).
KERNEL_FILES = ("lbm_lattice.cuh", "lbm_collide.cuh", "lbm_kernels.cuh", "lbm_step_d3q19.cu",
                "lbm_step_d2q9.cu", "lbm_internal.h")   # the last holds the launch shape


def ncu_traffic(workload: str, cells: int, src: str):
    """DRAM bytes per step launch for ``workload`` from NCU_TRAFFIC, or None when there is
    no figure or it was taken on kernel sources other than ``src`` (their hash)."""
    tr = NCU_TRAFFIC.get(workload)
    if not tr or tr["src_hash"] != src:
        return None
    return round(tr["bytes_per_cell"] * cells)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lattice_boltzmann_cfd_gb300", "csrc")
    for name in KERNEL_FILES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def make_workload(name: str):
    from lattice_boltzmann_cfd_gb300 import workloads as W
    table = {
        "d3q19_mrt_periodic_512": lambda: W.random_periodic(n=512, seed=2),
        "d3q19_mrt_periodic_256": lambda: W.random_periodic(n=256, seed=2),
        "d3q19_mrt_periodic_128": lambda: W.random_periodic(n=128, seed=2),
        # rows of 258 cells: the step kernels' 1-D launch over the cells
        "d3q19_mrt_periodic_258x256x256": lambda: W.random_periodic(shape=(258, 256, 256),
                                                                    seed=2),
        "cavity3d_256": lambda: W.cavity3d(n=256),
        "taylor_green_32": lambda: W.taylor_green(),
        "channel_sphere_128": lambda: W.channel_sphere(),
        "channel_ib_sphere_128": lambda: W.channel_ib_sphere(),
        "cavity2d_4096": lambda: W.cavity2d(),
        "cavity2d_2048": lambda: W.cavity2d(n=2048),
        "cavity3d_512": lambda: W.cavity3d(),
        "d3q27_cm_periodic_512": lambda: W.random_periodic(n=512, seed=2, lattice=27),
        "d3q27_cm_periodic_256": lambda: W.random_periodic(n=256, seed=2, lattice=27),
        "channel_sphere_d3q27_128": lambda: W.channel_sphere(lattice=27),
        "channel_ib_sphere_d3q27_128": lambda: W.channel_ib_sphere(lattice=27),
    }
    return table[name]()


def workload_label(name, w=None) -> str:
    return {
        "d3q19_mrt_periodic_512": "D3Q19 MRT periodic 512^3, seeded rho=1+N(0,1e-3), "
                                  "u~U(-0.02,0.02), nu=0.01, other rates 1.2",
        "d3q19_mrt_periodic_128": "D3Q19 MRT periodic 128^3, seeded rho=1+N(0,1e-3), "
                                  "u~U(-0.02,0.02), nu=0.01, other rates 1.2",
    }.get(name, w.name if w is not None else name)


# ------------------------------------------------------------------ clocks ---------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi clock samples every 200 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        sm = [r[0] for r in rows]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows),
                "reasons": reasons}


# ------------------------------------------------------------------ GPU legs -------

def upload(w, device, pinned=False):
    import torch
    arrs = [w.rho0, w.u0] + ([w.T_init] if w.thermal else [])
    out = []
    for a in arrs:
        t = torch.from_numpy(np.ascontiguousarray(a))
        out.append(t.pin_memory() if pinned else t.to(device))
    if not w.thermal:
        out.append(None)
    return out


def timed_device_leg(sim, w, steps, warmup, lbm_steps, dist_ctx):
    """K submissions on a device-resident state; returns (seconds, kernel_ms, clocks)."""
    import torch
    for _ in range(warmup):
        sim.step(lbm_steps)
        sim.diagnostics(allow_nonfinite=True)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        t0.record()
        for k in range(steps):
            ev[k][0].record()
            sim.step(lbm_steps)
            ev[k][1].record()
            sim.diagnostics(allow_nonfinite=True)
        t1.record()
        torch.cuda.synchronize()
    dist_ctx.barrier()
    secs = t0.elapsed_time(t1) / 1e3
    per_step = [a.elapsed_time(b) / lbm_steps for a, b in ev]   # ms per LBM step
    kernel_ms = sum(per_step) / steps
    return secs, kernel_ms, clk.summary(), per_step


def live_copy_gbs(nbytes: int = 2 << 30, reps: int = 5) -> float:
    """Device-to-device copy bandwidth measured now (read + write bytes / time): a second
    roofline denominator taken in the same run as the kernel."""
    import torch
    n = nbytes // 4
    a = torch.empty(n, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    a.fill_(1.0)
    for _ in range(2):
        b.copy_(a)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(reps):
        b.copy_(a)
    t1.record()
    torch.cuda.synchronize()
    gbs = 2 * nbytes * reps / (t0.elapsed_time(t1) / 1e3) / 1e9
    del a, b
    torch.cuda.empty_cache()
    return gbs


def nominal_hbm_gbs():
    """2 x memory clock x bus width of the current device, or None if neither torch's device
    properties nor (nvidia-smi's maximum memory clock, the CUDA runtime's bus-width
    attribute) give them."""
    import torch
    dev = torch.cuda.current_device()
    p = torch.cuda.get_device_properties(dev)
    clk_khz = getattr(p, "memory_clock_rate", None)
    bus = getattr(p, "memory_bus_width", None)
    if not clk_khz or not bus:
        try:
            q = subprocess.run(["nvidia-smi", "-i", str(dev), "--query-gpu=clocks.max.memory",
                                "--format=csv,noheader,nounits"], capture_output=True,
                               text=True, timeout=20)
            clk_khz = float(q.stdout.strip().splitlines()[0]) * 1e3
            import ctypes
            rt = None
            for name in ("libcudart.so", "libcudart.so.13", "libcudart.so.12"):
                try:
                    rt = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            v = ctypes.c_int(0)
            if rt is None or rt.cudaDeviceGetAttribute(ctypes.byref(v), 37, dev) != 0:
                return None            # 37 = cudaDevAttrGlobalMemoryBusWidth
            bus = v.value
        except (OSError, ValueError, IndexError, subprocess.SubprocessError):
            return None
    if not clk_khz or not bus:
        return None
    return 2.0 * clk_khz * 1e3 * bus / 8 / 1e9


def timed_e2e_leg(sim, w, steps, warmup, lbm_steps, dist_ctx):
    """K submissions through the C ABI with page-locked host fields."""
    import torch
    rho_h, u_h, T_h = upload(w, None, pinned=True)
    out_rho = torch.empty_like(rho_h).pin_memory()
    out_u = torch.empty_like(u_h).pin_memory()
    out_T = torch.empty_like(T_h).pin_memory() if T_h is not None else None

    def one():
        sim.init_equilibrium(rho_h, u_h, T_h)
        sim.step(lbm_steps)
        sim.macroscopic(out_rho, out_u, out_T)
        sim.diagnostics(allow_nonfinite=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        one()
    t1.record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    secs = t0.elapsed_time(t1) / 1e3
    h2d = sum(t.numel() * t.element_size() for t in (rho_h, u_h, T_h) if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in (out_rho, out_u, out_T) if t is not None)
    d2h += 18 * 8   # diagnostics read-back
    return secs, h2d, d2h


def timed_pipelined_e2e_leg(sim, w, steps, warmup, lbm_steps, dist_ctx):
    """The same jobs through JobPipeline: each job's host-to-device copy and read-out still
    happen inside the timed region; the next job's upload travels beside the steps."""
    import torch
    from lattice_boltzmann_cfd_gb300.pipeline import JobPipeline
    rho_h, u_h, T_h = upload(w, None, pinned=True)
    outs = tuple(None if t is None else torch.empty_like(t).pin_memory()
                 for t in (rho_h, u_h, T_h))
    pipe = JobPipeline(sim)
    job = ((rho_h, u_h, T_h), outs)
    pipe.run([job] * warmup, lbm_steps)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(pipe.compute)
    pipe.h2d.wait_event(t0)
    pipe.run([job] * steps, lbm_steps)
    pipe.compute.wait_stream(pipe.d2h)
    t1.record(pipe.compute)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    return t0.elapsed_time(t1) / 1e3


# --------------------------------------------------------------- CPU baseline ------

def oracle_sample(name: str):
    """A bounded sample of the workload for the CPU oracle: the same generator and
    physics on a smaller grid (periodic sub-box / reduced cavity)."""
    from lattice_boltzmann_cfd_gb300 import workloads as W
    if name.startswith("d3q19_mrt_periodic"):
        return W.random_periodic(shape=(512, 512, 64), seed=2), "periodic 512x512x64 slab"
    if name.startswith("cavity3d"):
        return W.cavity3d(shape=(512, 512, 48)), "cavity 512x512x48 slab"
    if name == "cavity2d_4096":
        return W.cavity2d(shape=(2048, 2048, 1)), "cavity 2048^2"
    if name == "channel_sphere_128":
        return W.channel_sphere(), "full 128^3"
    return W.taylor_green(), "full 32^3"


def time_oracle(name: str, steps: int):
    import oracle
    oracle.build()
    w, label = oracle_sample(name)
    p = oracle.Problem(w)
    f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    oracle.run(p, f, g, 1)   # first touch
    t = time.perf_counter()
    oracle.run(p, f, g, steps)
    dt = time.perf_counter() - t
    mlups = w.cells * steps / dt / 1e6
    return mlups, dt, w.cells, label, oracle.max_threads()


def cpu_baseline(name: str, steps: int = 16, steps_1thread: int = 1) -> dict:
    import oracle
    mlups, dt, cells, label, cores = time_oracle(name, steps)
    prev = oracle.set_threads(1)
    try:
        mlups1, dt1, _, _, _ = time_oracle(name, steps_1thread)
    finally:
        oracle.set_threads(prev)
    return {"value": round(mlups, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{label} of the same workload, {steps} fp64 two-buffer steps "
                      f"({cells * steps / 1e6:.0f} M cell updates, {dt:.1f} s)",
            "value_1thread": round(mlups1, 3),
            "sample_1thread": f"the same sample, {steps_1thread} steps on 1 thread "
                              f"({dt1:.1f} s)"}


# ----------------------------------------------------------------- helpers --------

class DistCtx:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def done(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


_WORKLOAD_CACHE = {}


def cached_workload(name):
    if name not in _WORKLOAD_CACHE:
        _WORKLOAD_CACHE[name] = make_workload(name)
    return _WORKLOAD_CACHE[name]


def run_secondary(name, lbm_steps, reps, streaming="aa"):
    """Kernel-only MLUPS of a workload in one population layout ("aa", "pull", "split")."""
    import torch
    from lattice_boltzmann_cfd_gb300 import Simulation
    w = cached_workload(name)
    sim = Simulation(w, streaming=streaming)
    sim.init_equilibrium(*upload(w, sim.device))
    sim.step(lbm_steps)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        sim.step(lbm_steps)
    b.record()
    torch.cuda.synchronize()
    kernel_s = a.elapsed_time(b) / 1e3 / (reps * lbm_steps)
    bpc = BYTES_PER_CELL[(w.lattice, w.thermal)] * (2 if streaming == "split" else 1)
    peak, _ = measured_peak()
    achieved = bpc * w.cells / kernel_s / 1e9
    sim.close()
    del sim
    torch.cuda.empty_cache()
    out = {"workload": workload_label(name, w), "layout": streaming,
           "mlups": round(w.cells / kernel_s / 1e6, 1),
           "bytes_per_cell": bpc, "achieved_gbs": round(achieved, 1),
           "frac": round(achieved / peak, 4)}
    if w.solid is not None:   # fluid cells only (solid cells are skipped, not updated)
        out["fluid_mlups"] = round(w.fluid_cells() / kernel_s / 1e6, 1)
    return out


def run_moving_ib_secondary(name, lbm_steps, reps):
    """The immersed-boundary channel with its samples replaced before every step from
    device tensors (lbm_set_ib_samples_device: placement, radix sort by l-block and Morton
    code, re-marking of the stencils, all on the device), against the same steps with the
    samples left in place.  The positions of every step are prepared before the timed
    region (a sphere translating by 0.01 cells per step)."""
    import torch
    from lattice_boltzmann_cfd_gb300 import Simulation
    w = cached_workload(name)
    sim = Simulation(w)
    sim.init_equilibrium(*upload(w, sim.device))
    x0 = torch.from_numpy(w.ib_x).to(sim.device)
    v = torch.tensor([0.01, 0.0, 0.0], device=sim.device)
    X = torch.stack([x0 + k * v for k in range(lbm_steps)]).contiguous()
    ub = torch.zeros_like(x0)
    ub[:, 0] = 0.01
    wt = torch.from_numpy(w.ib_w).to(sim.device)
    sim.step(4)
    torch.cuda.synchronize()

    def timed(mode):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sim.set_ib_samples_device(X[0], ub, wt, reorder=True)
        a.record()
        for _ in range(reps):
            for k in range(lbm_steps):
                if mode != "static":
                    sim.set_ib_samples_device(X[k], ub, wt, reorder=(mode == "sort"))
                sim.step(1)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * lbm_steps)

    timed("sort")
    static_ms, keep_ms, sort_ms = timed("static"), timed("keep"), timed("sort")
    sim.close()
    del sim
    torch.cuda.empty_cache()
    return {"workload": workload_label(name, w) + ", samples replaced every step",
            "layout": "aa", "samples": int(len(w.ib_x)),
            "ms_per_step_static": round(static_ms, 4),
            "ms_per_step_moving": round(keep_ms, 4),
            "ms_per_step_moving_resorted": round(sort_ms, 4),
            "mlups": round(w.cells / (keep_ms / 1e3) / 1e6, 1),
            "update_us": round((keep_ms - static_ms) * 1e3, 2),
            "update_us_resorted": round((sort_ms - static_ms) * 1e3, 2),
            "moving": "lbm_set_ib_samples_device before every step in the stored order of "
                      "one sort (update_us), or sorted every step (update_us_resorted)"}


def run_slabs_secondary(name, nslabs, lbm_steps, reps, single_mlups=None, overlap=False):
    """MLUPS of a workload run as ``nslabs`` slabs along its outer axis on this GPU, with
    the halo exchange after every step (a step = one step launch per slab + the exchange's
    pack and unpack launches).  overlap: interior planes, boundary planes, and the exchange
    on a second stream beside the next step's interior (two step launches per slab)."""
    import torch
    from lattice_boltzmann_cfd_gb300.slabs import SlabDomain
    w = cached_workload(name)
    dom = SlabDomain(w, nslabs, overlap=overlap)
    dom.init_equilibrium()
    dom.step(4)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dom.step(lbm_steps)
    b.record()
    torch.cuda.synchronize()
    step_s = a.elapsed_time(b) / 1e3 / (reps * lbm_steps)
    halo = dom.halo_bytes_per_step()
    launches = (len(dom.pairs()) + 31) // 32 if dom.swap else 4 * len(dom.pairs())
    dom.close()
    del dom
    torch.cuda.empty_cache()
    mlups = w.cells / step_s / 1e6
    out = {"workload": workload_label(name, w), "layout": "aa", "slabs": nslabs,
           "decomposition": "slabs along the outer axis, 1 ghost plane per inner face, "
                            "FILL after even / DRAIN after odd steps, all on this GPU, every "
                            "face moved by one buffer-free swap launch",
           "overlap": bool(overlap),
           "mlups": round(mlups, 1), "halo_bytes_per_step": int(halo),
           "halo_launches_per_step": launches}
    if single_mlups:
        out["vs_single_domain"] = round(mlups / single_mlups, 4)
    return out


def run_blocks_secondary(name, nb, lbm_steps, reps, single_mlups=None, overlap=False):
    """MLUPS of a workload cut into nb = (bx, by, bz) blocks on this GPU, with the per-axis
    halo exchange after every step (z, then y, then x; a step = one step launch per block +
    one pack and one unpack launch per block face and direction)."""
    import torch
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    w = cached_workload(name)
    dom = BlockDomain(w, nb, overlap=overlap)
    dom.init_equilibrium()
    dom.step(4)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dom.step(lbm_steps)
    b.record()
    torch.cuda.synchronize()
    step_s = a.elapsed_time(b) / 1e3 / (reps * lbm_steps)
    halo = dom.halo_bytes_per_step()
    launches = dom.halo_launches_per_step()
    dom.close()
    del dom
    torch.cuda.empty_cache()
    mlups = w.cells / step_s / 1e6
    out = {"workload": workload_label(name, w), "layout": "aa", "blocks": list(nb),
           "decomposition": "blocks, 1 ghost plane per inner face of each split axis, "
                            "exchanged axis by axis with the ghost rows of the other axes "
                            "(edges and corners in two or three hops), all on this GPU, the "
                            "faces of each axis moved by one buffer-free swap launch",
           "overlap": bool(overlap),
           "mlups": round(mlups, 1), "halo_bytes_per_step": int(halo),
           "halo_launches_per_step": launches}
    if single_mlups:
        out["vs_single_domain"] = round(mlups / single_mlups, 4)
    return out


# --------------------------------------------------------------------- main --------

def run_gpu(args, dctx):
    import torch
    from lattice_boltzmann_cfd_gb300 import Simulation, capi
    torch.cuda.set_device(dctx.local)
    dctx.init("nccl")
    capi.load()
    w = make_workload(args.workload)
    sim = Simulation(w)
    sim.init_equilibrium(*upload(w, sim.device))
    secs, kernel_ms, clocks, per_step = timed_device_leg(sim, w, args.steps, args.warmup,
                                                         args.lbm_steps, dctx)
    secs = dctx.max(secs)
    kernel_ms = dctx.max(kernel_ms)
    updates = w.cells * args.lbm_steps * args.steps * dctx.world
    value = updates / secs / 1e6
    e2e_secs, h2d, d2h = timed_e2e_leg(sim, w, args.steps, min(args.warmup, 2),
                                       args.lbm_steps, dctx)
    e2e_secs = dctx.max(e2e_secs)
    e2e_value = updates / e2e_secs / 1e6
    pipe_secs = dctx.max(timed_pipelined_e2e_leg(sim, w, args.steps, min(args.warmup, 2),
                                                 args.lbm_steps, dctx))
    pipelined_value = updates / pipe_secs / 1e6
    sim.close()
    del sim
    torch.cuda.empty_cache()
    if dctx.rank != 0:
        return None
    bpc = BYTES_PER_CELL[(w.lattice, w.thermal)]
    peak, peak_kind = measured_peak()
    achieved = bpc * w.cells / (kernel_ms / 1e3) / 1e9
    live = live_copy_gbs()
    nominal = nominal_hbm_gbs()
    per_step = sorted(per_step)
    median_ms = per_step[len(per_step) // 2] if len(per_step) % 2 else \
        0.5 * (per_step[len(per_step) // 2 - 1] + per_step[len(per_step) // 2])
    src = kernel_source_hash()
    tr = NCU_TRAFFIC.get(args.workload)
    traffic = ncu_traffic(args.workload, w.cells, src)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dctx.world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_label(args.workload, w),
                   "grid": list(w.shape), "cells": w.cells,
                   "lbm_steps_per_step": args.lbm_steps,
                   "step": f"{args.lbm_steps} fused AA collide-and-stream launches + "
                           "diagnostics reduction read back",
                   "layout": "AA in-place, one fp32 SoA population buffer",
                   "streaming": "aa",
                   "l2": "state far larger than the 129 MB L2 (no flush needed)",
                   "parallelism": f"replicas x{dctx.world}" if dctx.world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel_src_hash": src,
                     "traffic_src_hash": tr["src_hash"] if tr else None,
                     # the counters' figure, for sources other than these when traffic is null
                     "traffic_last_measured": (round(tr["bytes_per_cell"] * w.cells)
                                               if tr else None),
                     "kernel": "step_kernel (even/odd AA forms)",
                     "kernel_ms": round(kernel_ms, 4), "bytes_per_cell": bpc,
                     "kernel_ms_median": round(median_ms, 4),
                     "kernel_ms_mean": round(kernel_ms, 4),
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json)",
                     "live_copy_gbs": round(live, 1),
                     "frac_of_live_copy": round(achieved / live, 4),
                     "nominal_gbs": None if nominal is None else round(nominal, 1),
                     "frac_of_nominal": None if nominal is None else round(achieved / nominal, 4),
                     "denominators": "peak: the measured copy; live_copy_gbs: a 2 GiB "
                                     "device copy timed in this run; nominal: 2 x memory "
                                     "clock x bus width from the device attributes"},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "path": "one step at a time through the C ABI: lbm_init_equilibrium reads "
                        "the page-locked host rho,u, lbm_step, lbm_macroscopic writes "
                        "page-locked host fields, lbm_diagnostics",
                "pipelined_value": round(pipelined_value, 1),
                "pipelined": "the same steps through JobPipeline: the next step's upload "
                             "in ~32 MB pieces on a copy stream beside the LBM steps, the "
                             "read-out written to host by lbm_macroscopic; 31-39k MLUPS "
                             "between runs, so value is the serial path"},
        "gpu_launches": args.steps * (args.lbm_steps + 2),
        "clocks": clocks,
    }
    if not args.no_secondary:
        _WORKLOAD_CACHE[args.workload] = w
        line["secondary"] = []

        def secondary(fn, *a):
            """One secondary measurement; an error there is recorded in its entry instead of
            ending the run (the headline line above does not depend on it)."""
            try:
                line["secondary"].append(fn(*a))
            except Exception as e:   # noqa: BLE001 -- report any failure, keep the headline
                line["secondary"].append({"run": f"{fn.__name__}{a[:2]}",
                                          "error": f"{type(e).__name__}: {e}"[:300]})
                import torch
                torch.cuda.synchronize()
                torch.cuda.empty_cache()

        runs = [("cavity3d_512", "aa"), ("cavity2d_4096", "aa"), ("taylor_green_32", "aa"),
                ("channel_ib_sphere_128", "aa"), ("d3q27_cm_periodic_512", "aa"),
                ("channel_sphere_d3q27_128", "aa"), ("channel_ib_sphere_d3q27_128", "aa")]
        # the streaming-layout page's comparison: in place vs two buffers
        for n in ("d3q19_mrt_periodic_128", "channel_sphere_128", args.workload):
            runs += [(n, "aa"), (n, "pull"), (n, "split")]
        for n, mode in runs:
            if n == args.workload and mode == "aa":
                continue
            # the 32^3 case fits in L2 and is launch-bound: long submissions replay graphs
            steps_n = 2048 if n == "taylor_green_32" else args.lbm_steps
            secondary(run_secondary, n, steps_n, 4, mode)
        secondary(run_moving_ib_secondary, "channel_ib_sphere_128", args.lbm_steps, 4)
        single = {r["workload"]: r["mlups"] for r in line["secondary"]
                  if r.get("layout") == "aa" and "mlups" in r}
        # the steps alone, as the secondaries time them (value adds the diagnostics)
        single[workload_label(args.workload, w)] = round(w.cells / (kernel_ms / 1e3) / 1e6, 1)
        for n in (args.workload, "cavity3d_512"):
            lbl = workload_label(n, cached_workload(n))
            for overlap in (False, True):
                secondary(run_slabs_secondary, n, 4, args.lbm_steps, 2, single.get(lbl),
                          overlap)
            for nb, overlap in (((1, 2, 2), False), ((1, 2, 2), True), ((1, 2, 4), False)):
                secondary(run_blocks_secondary, n, nb, args.lbm_steps, 2, single.get(lbl),
                          overlap)
        lbl = workload_label("cavity2d_4096", cached_workload("cavity2d_4096"))
        secondary(run_blocks_secondary, "cavity2d_4096", (2, 2, 1), args.lbm_steps, 2,
                  single.get(lbl))
    line["cpu_baseline"] = cpu_baseline(args.workload)
    return line


def run_reference(args, dctx):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    if dctx.rank != 0:
        return None
    import oracle
    oracle.build()
    w, label = oracle_sample(args.workload)
    p = oracle.Problem(w)
    f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    for _ in range(args.warmup):
        oracle.run(p, f, g, 1)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(p, f, g, 1)
    dt = time.perf_counter() - t
    value = w.cells * args.steps / dt / 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": dctx.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(args.workload),
                   "sample": label, "lbm_steps_per_step": 1},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{label}: one fp64 two-buffer step per benchmark step"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="d3q19_mrt_periodic_512")
    ap.add_argument("--lbm-steps", type=int, default=50,
                    help="time steps per benchmark step (one submission)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="do not measure the other workloads after the main one")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dctx = DistCtx()
    line = run_reference(args, dctx) if args.impl == "reference" else run_gpu(args, dctx)
    if line is not None:
        print(json.dumps(line), flush=True)
    dctx.done()


if __name__ == "__main__":
    main()
