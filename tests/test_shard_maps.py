"""Host-side row maps of the sharded path: every row of every table is owned by
exactly one rank, in both maps, and the local tables the ranks build match the
rows they own."""
import numpy as np
import pytest

from sparse_embedding_bag_gb300 import shard as S


@pytest.mark.parametrize("cyclic", [False, True])
@pytest.mark.parametrize("world", [1, 3, 8])
def test_every_row_owned_once(cyclic, world):
    rows, dims = [97, 8, 1000, 5], [4, 8, 16, 4]
    rb = S.even_row_bounds(rows, world)
    assert rb.shape == (4, world + 1) and np.all(rb[:, 0] == 0) and np.all(rb[:, -1] == rows)
    assert np.all(np.diff(rb, axis=1) >= 0)
    seen = [np.zeros(r, int) for r in rows]
    for r in range(world):
        own = S.owned_rows(rows, rb, r, world, cyclic)
        local, hsc, Do, wo = S.local_tables(rows, dims, rb, r, world, cyclic)
        for t in range(len(rows)):
            seen[t][own[t]] += 1
            assert own[t].size == local[t]
            if cyclic:  # local row k is global row k * W + r
                assert np.array_equal(own[t], np.arange(local[t]) * world + r)
        assert np.array_equal(hsc, np.concatenate([[0], np.cumsum(local)]))
        assert np.array_equal(Do, np.concatenate([[0], np.cumsum(dims)]))
        assert np.array_equal(wo, np.concatenate([[0], np.cumsum(local * np.array(dims))[:-1]]))
    assert all(np.all(s == 1) for s in seen)
