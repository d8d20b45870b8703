"""Host-side logic of bench.py that needs no GPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("n", list(range(0, 30)) + [100, 257])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_e2e_groups_cover_every_step_once(n, group):
    sizes = bench.e2e_group_sizes(n, group)
    assert sum(sizes) == n
    assert all(1 <= s <= group for s in sizes) or (group == 1 and all(s == 1 for s in sizes))
    if n >= 3:
        # nothing overlaps the first group's input copy or the last group's output copy
        assert sizes[0] == 1 and sizes[-1] == 1
        # every group between them is full except at most one
        assert sum(1 for s in sizes[1:-1] if s != group) <= 1


def test_e2e_groups_of_the_default_run():
    assert bench.e2e_group_sizes(20, 4) == [1, 4, 4, 4, 4, 2, 1]
