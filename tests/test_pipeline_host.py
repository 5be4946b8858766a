"""Host logic of JobPipeline that needs no GPU."""
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
