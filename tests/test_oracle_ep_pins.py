"""Pins for the oracle's expert-parallel receive-side map (no GPU).

"02 · DeepSeek-V3" (PaperTrace) §1.3 / §5.1: experts are partitioned across
devices and each device runs its local experts on the rows it receives.  The
rows arrive source by source (each source's rows sorted by expert); the map
regroups them expert by expert, sources in order, keeping each block's row
order.  Pinned by a worked example, by brute force (sorting row labels) and
by the map's invariants."""
import numpy as np
import pytest

from oracle import moe_oracle as O


def test_worked_example():
    # source 0 sends 1 row to expert 0 and 2 to expert 1; source 1 sends 3
    # rows to expert 0.  Source-major: (0,0,0) (0,1,0) (0,1,1) (1,0,0)
    # (1,0,1) (1,0,2); expert-major: expert 0 = (0,0,0) (1,0,*), then
    # expert 1 = (0,1,*).
    perm, off = O.ep_plan(np.array([[1, 2], [3, 0]]))
    assert perm.tolist() == [0, 4, 5, 1, 2, 3]
    assert off.tolist() == [0, 4, 6]


@pytest.mark.parametrize("P,El,seed", [(2, 3, 0), (8, 32, 1), (3, 1, 2),
                                       (1, 5, 3), (4, 4, 4)])
def test_brute_force_against_sorted_labels(P, El, seed):
    rng = np.random.default_rng(seed)
    rc = rng.integers(0, 5, (P, El))
    rc[rng.random((P, El)) < 0.2] = 0       # empty blocks
    labels = [(s, l, j) for s in range(P) for l in range(El)
              for j in range(rc[s, l])]
    order = sorted(range(len(labels)),
                   key=lambda i: (labels[i][1], labels[i][0], labels[i][2]))
    want = np.empty(len(labels), np.int64)
    want[order] = np.arange(len(labels))
    perm, off = O.ep_plan(rc)
    assert np.array_equal(perm, want)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(rc.sum(0))]))


def test_map_is_a_bijection_that_groups_by_expert():
    rng = np.random.default_rng(7)
    rc = rng.integers(0, 40, (8, 32))
    perm, off = O.ep_plan(rc)
    rows = int(rc.sum())
    assert np.array_equal(np.sort(perm), np.arange(rows))
    expert_of_src_row = np.repeat(np.tile(np.arange(32), 8), rc.ravel())
    grouped = np.empty(rows, np.int64)
    grouped[perm] = expert_of_src_row
    # expert-major: experts ascending, segment l = [off[l], off[l+1])
    assert np.all(np.diff(grouped) >= 0)
    for l in range(32):
        assert np.all(grouped[off[l]:off[l + 1]] == l)
    # inverse round trip
    x = rng.standard_normal(rows)
    y = np.empty_like(x)
    y[perm] = x
    assert np.array_equal(y[perm], x)


def test_no_rows():
    perm, off = O.ep_plan(np.zeros((3, 4), np.int64))
    assert perm.size == 0 and off.tolist() == [0] * 5
