"""Head-group layout of the host pipeline (pure host logic, CPU only)."""
import pytest

from precision_numerics_gb300.host import ramped_group_sizes


@pytest.mark.parametrize("bh,chunks", [(32, 4), (96, 4), (24, 4), (12, 6), (64, 8)])
def test_half_groups_at_both_ends(bh, chunks):
    m = bh // chunks
    assert ramped_group_sizes(bh, chunks) == [m // 2] + [m] * (chunks - 1) + [m // 2]


@pytest.mark.parametrize("bh", [1, 2, 3, 5, 7, 31, 32, 33, 100, 70000])
@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 7, 64])
def test_sizes_cover_every_head_once(bh, chunks):
    g = ramped_group_sizes(bh, chunks)
    assert sum(g) == bh
    assert all(x >= 1 for x in g)
    assert len(g) <= min(bh, chunks + 1)


def test_rejects_empty_problem():
    with pytest.raises(ValueError):
        ramped_group_sizes(0, 4)
