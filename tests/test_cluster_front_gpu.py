"""GPU parity of the small-batch front (one cluster of CTAs per table sorts and
run-length encodes the table's lookups in one launch).

Both fronts sort each table's lookups stably on the row index, so every call
must give the oracle's integer outputs bit for bit (sorted unique keys, run
lengths and starts, long runs as a set) and, fed to the same reduce, bitwise
identical weights and state. Each case runs on two plans of the same workload,
one of them created with EMB_FLAG_NO_CLUSTER_FRONT, and is compared with the
oracle as in the other parity tests.
"""
import numpy as np
import pytest

from _helpers import compare_momentum, compare_runs, compare_weights, oracle_step
import oracle
from sparse_embedding_bag_gb300 import device as dev
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_embedding_bag_gb300 import build
    build.build()
    E.load()


def custom(seed, rows, dims, B, lengths_fn, ids_fn=None, **kw):
    rng = np.random.default_rng(seed + 5000)
    lengths = lengths_fn(rng, len(rows), B)
    ids_fn = ids_fn or (lambda r, t, n: synth.sample_zipf(r, rows[t], 1.05, n))
    return synth.make_bag_workload("custom", seed, rows, dims, B, lengths, ids_fn, **kw)


def run_front(w, flags, thr=0):
    """One step on a fresh device copy; returns (weights, momentum, runs, stage times)."""
    dw = dev.to_device(w)
    plan = dev.make_plan(w, max_segment_length_per_warp=thr, flags=flags)
    try:
        E.emb_plan_set_profiling(plan, True)
        dev.step(plan, dw)
        assert E.emb_plan_status(plan) == E.EMB_OK
        runs = E.emb_plan_debug_runs(plan, max(w.N, 1))
        ms = E.emb_plan_stage_ms(plan)
    finally:
        E.emb_plan_destroy(plan)
    m = None if dw.momentum is None else dw.momentum.cpu().numpy()
    return dev.weights_numpy(dw), m, runs, ms


def check_both_fronts(w, thr=0, expect_cluster=True):
    """expect_cluster: True, the default plan takes the small-batch front; False,
    the multi-block one; None, either."""
    wc, mc, rc, msc = run_front(w, 0, thr)
    wb, mb, rb, msb = run_front(w, E.EMB_FLAG_NO_CLUSTER_FRONT, thr)
    exp = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, thr or 32)
    compare_runs(rc, exp)
    compare_runs(rb, exp)
    # the long runs are listed in key order by both fronts
    np.testing.assert_array_equal(rc["long_ids"], rb["long_ids"])
    bits = np.uint32 if wc.dtype == np.float32 else np.uint16
    assert np.array_equal(wc.view(bits), wb.view(bits)), "the two fronts disagree on the weights"
    if mc is not None:
        assert np.array_equal(mc.view(np.uint32), mb.view(np.uint32)), "the two fronts disagree on the state"
    # the small-batch front is one launch: its sort and run-length stages are
    # empty (back-to-back events, a few microseconds at most)
    if expect_cluster:
        assert msc[1] + msc[2] < 0.006, msc
    elif expect_cluster is not None:  # the multi-block front: a radix-sort stage of its own
        assert msc[1] > 0.006, msc
    assert msb[1] > 0.0, msb
    ew, em = oracle_step(w)
    compare_weights(w, wc, ew, exp["run_keys"])
    if em is not None:
        compare_momentum(w, mc, em)


def test_dlrm_like():
    # the DLRM-like recipe (8 tables x 100k rows, D=64, Zipf(1.05), row-wise
    # Adagrad) at a batch the small-batch front takes
    w = custom(10, [100_000] * 8, [64] * 8, 512, lambda r, T, B: r.integers(1, 21, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    assert 20_000 < w.N <= 1 << 16
    check_both_fronts(w)


def test_dlrm_full_batch_takes_the_multiblock_front():
    w = synth.dlrm(3)
    assert w.N > 1 << 16
    check_both_fronts(w, expect_cluster=False)


def test_lm_unpooled():
    check_both_fronts(synth.lm(1))


def test_tiny():
    check_both_fronts(synth.tiny(2))


@pytest.mark.parametrize("opt", [synth.SGD, synth.ROWWISE_ADAGRAD])
@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.SUM, True), (synth.MEAN, True)])
def test_row_widths_and_payloads(opt, pooling, weighted):
    # several team shapes (segments of tables), 64-bit payloads when weighted or mean
    w = custom(1, [3000, 500, 20000, 70, 9000], [8, 64, 128, 256, 32], 700,
               lambda r, T, B: r.integers(0, 25, (T, B)), optimizer=opt, pooling=pooling,
               weighted=weighted, weight_dtype=synth.F16,
               momentum_init=0.5 if opt == synth.ROWWISE_ADAGRAD else 0.0)
    check_both_fronts(w)


def test_one_table_holds_most_lookups():
    # table 1 holds ~95 % of the batch: its CTAs' slices are near their capacity,
    # the other tables' slices nearly empty
    def lengths(r, T, B):
        L = r.integers(0, 3, (T, B))
        L[1] = r.integers(40, 80, B)
        return L
    w = custom(2, [400, 60000, 900], [16, 16, 16], 1000, lengths, optimizer=synth.ROWWISE_ADAGRAD)
    assert 50000 < w.N <= 1 << 16
    check_both_fronts(w)


def test_empty_tables():
    # tables with no lookups at the start, in the middle and at the end
    def lengths(r, T, B):
        L = r.integers(0, 12, (T, B))
        L[0] = 0
        L[2] = 0
        L[T - 1] = 0
        return L
    w = custom(3, [100, 5000, 700, 3000, 50], [16, 32, 32, 64, 64], 300, lengths,
               optimizer=synth.ROWWISE_ADAGRAD)
    check_both_fronts(w)


def test_empty_bags_and_tiny_tables():
    w = custom(4, [1, 2, 3, 4000], [4, 8, 4, 16], 200,
               lambda r, T, B: r.integers(0, 3, (T, B)) * (r.random((T, B)) < 0.5))
    check_both_fronts(w)


@pytest.mark.parametrize("rows", [[600], [150_000, 150_000], [(1 << 20) + 5], [(1 << 24) + 3]])
def test_passes(rows):
    # row widths of 10 to 25 bits: one to three radix passes of up to 9 bits
    w = custom(5 + rows[0] % 97, rows, [4] * len(rows), 800, lambda r, T, B: r.integers(0, 30, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.5, synth.sample_zipf(r, rows[t], 1.05, n),
                                               r.integers(0, rows[t], n)))
    check_both_fronts(w)


@pytest.mark.parametrize("thr", [1, 7, 1000])
def test_thresholds(thr):
    w = custom(6, [2000, 300], [16, 32], 1000, lambda r, T, B: r.integers(0, 20, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    check_both_fronts(w, thr=thr)


def test_hot_row_across_all_slices():
    # one row takes 60 % of a table's lookups: its run spans every CTA's slice
    w = custom(7, [5000], [64], 3000, lambda r, T, B: r.integers(1, 20, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.6, 17, r.integers(0, 5000, n)).astype(np.int64),
               optimizer=synth.ROWWISE_ADAGRAD)
    check_both_fronts(w)


def test_many_tables():
    # more tables: clusters of 8 CTAs where 16 no longer fit at once, or the other front
    rows = [500 + 37 * t for t in range(14)]
    w = custom(8, rows, [16] * 14, 400, lambda r, T, B: r.integers(0, 10, (T, B)))
    check_both_fronts(w, expect_cluster=None)


def test_largest_small_batch():
    # 2^16 lookups: the largest batch the small-batch front takes
    B = 1 << 13
    w = custom(9, [100_000, 100_000], [16, 16], B, lambda r, T, B: np.full((T, B), 4))
    assert w.N == 1 << 16
    check_both_fronts(w)
