"""Host logic of HostPipeline's head groups (no GPU): the groups partition
the heads in order, end groups are tapered, explicit sizes are validated."""
import pytest

from packed_sequence_attention_gb300 import head_groups


@pytest.mark.parametrize("n,g", [(42, 6), (42, 5), (42, 1), (42, 42), (9, 4), (7, 6), (13, 6),
                                 (16, 6), (1, 6), (100, 8)])
def test_groups_partition_the_heads_in_order(n, g):
    gr = head_groups(n, g)
    assert gr[0][0] == 0 and gr[-1][1] == n
    assert all(a < b for a, b in gr)
    assert all(gr[i][1] == gr[i + 1][0] for i in range(len(gr) - 1))
    assert max(b - a for a, b in gr) <= max(1, min(g, n))


def test_end_groups_are_tapered():
    assert [b - a for a, b in head_groups(42, 6)] == [3, 6, 6, 6, 6, 6, 6, 3]
    assert [b - a for a, b in head_groups(100, 8)] == [4] + [8] * 8 + [7] * 4 + [4]
    assert [b - a for a, b in head_groups(13, 6)] == [3, 4, 3, 3]
    assert [b - a for a, b in head_groups(42, 1)] == [1] * 42
    # too few heads for a taper: plain groups
    assert [b - a for a, b in head_groups(12, 6)] == [6, 6]
    assert [b - a for a, b in head_groups(42, 42)] == [42]


def test_explicit_group_sizes():
    assert head_groups(5, group_sizes=[1, 3, 1]) == [(0, 1), (1, 4), (4, 5)]
    for bad in ([1, 3], [0, 5], [6, -1], []):
        with pytest.raises(ValueError):
            head_groups(5, group_sizes=bad)
