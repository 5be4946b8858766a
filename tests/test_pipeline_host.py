"""Host logic that needs no GPU: JobPipeline's job checks and pieces, and the bench's
provenance rule for ncu traffic."""
from lattice_boltzmann_cfd_gb300.pipeline import _pieces


def test_pipeline_pieces_cover_every_element():
    """The pieces the copies and the step groups are cut into tile their range exactly,
    in order, for any piece count (empty pieces where there are fewer items than pieces)."""
    for n in (0, 1, 7, 50, 1000, 4097):
        for parts in (1, 2, 3, 50, 5000):
            p = _pieces(n, parts)
            assert len(p) == parts and p[0][0] == 0 and p[-1][1] == n
            assert all(a <= b for a, b in p)
            assert all(p[i][1] == p[i + 1][0] for i in range(parts - 1))
            sizes = [b - a for a, b in p]
            assert max(sizes) - min(sizes) <= 1


def test_check_jobs_accepts_the_workloads_fields():
    """Inputs and outputs shaped as the workloads build them pass, thermal or not, 2-D or
    3-D, with outputs None or with None entries."""
    import numpy as np
    from lattice_boltzmann_cfd_gb300 import workloads as W
    from lattice_boltzmann_cfd_gb300.pipeline import check_jobs
    for w in (W.cavity2d(shape=(96, 80, 1)), W.cavity3d(shape=(48, 20, 18)),
              W.random_periodic(shape=(64, 24, 20), seed=3)):
        grid, dim = w.rho0.shape, w.u0.shape[0]
        ins = (w.rho0, w.u0, w.T_init if w.thermal else None)
        outs = tuple(None if a is None else np.empty_like(a) for a in ins)
        check_jobs([(ins, outs), (ins, None), (ins, (outs[0], None, None))], grid, dim,
                   bool(w.thermal))


def test_check_jobs_rejects_malformed_jobs():
    """A missing or surplus temperature, a wrong shape or a malformed job raises before
    anything is launched."""
    import numpy as np
    import pytest
    from lattice_boltzmann_cfd_gb300.pipeline import check_jobs
    grid = (4, 5, 6)
    rho, u, T = np.zeros(grid), np.zeros((3,) + grid), np.zeros(grid)
    bad = [
        ([((rho, u, None), None)], True, "T is required"),
        ([((rho, u, T), None)], False, "given for a lattice without it"),
        ([((None, u, None), None)], False, "rho is required"),
        ([((rho, np.zeros((2,) + grid), None), None)], False, "input u has shape"),
        ([((rho, u, None), (np.zeros((4, 5, 7)), None, None))], False, "output rho has shape"),
        ([((rho, u, None),)], False, "expected (inputs, outputs)"),
        ([((rho, u), None)], False, "inputs must be"),
        ([((rho, u, None), (rho, u))], False, "outputs must be"),
    ]
    for jobs, thermal, msg in bad:
        with pytest.raises(ValueError, match=msg.replace("(", r"\(").replace(")", r"\)")):
            check_jobs(jobs, grid, 3, thermal)


def test_bench_reports_ncu_traffic_only_for_the_sources_it_was_taken_on():
    """The bench's roofline traffic comes from ncu counters tied to a hash of the kernel
    sources: the stored figure (bytes per cell x cells) while the hash matches, None once
    the sources differ or for a workload without a figure."""
    import bench
    w = "d3q19_mrt_periodic_512"
    tr = bench.NCU_TRAFFIC[w]
    cells = 512 ** 3
    assert bench.ncu_traffic(w, cells, tr["src_hash"]) == round(tr["bytes_per_cell"] * cells)
    assert bench.ncu_traffic(w, cells, "0" * 16) is None
    assert bench.ncu_traffic("no_such_workload", cells, tr["src_hash"]) is None
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    # every stored figure is positive and at most the algorithmic bytes (nothing re-read)
    lattices = {"d3q19_mrt_periodic_512": (19, 0), "cavity3d_512": (19, 7)}
    assert set(bench.NCU_TRAFFIC) == set(lattices)
    for name, t in bench.NCU_TRAFFIC.items():
        assert 0 < t["bytes_per_cell"] <= bench.BYTES_PER_CELL[lattices[name]]
