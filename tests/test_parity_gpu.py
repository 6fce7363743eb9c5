"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element on the same seeded inputs.

Bars: integer outputs (sorted unique linear indices, run lengths, cumulative
run lengths, number of runs) bit-exact, long-run ids as a set; fp32 weights and
momentum within rtol 1e-4 / atol 1e-5; fp16/bf16 weights within 1 ulp of the
oracle's round-to-nearest-even result; untouched rows bit-identical.
"""
import numpy as np
import pytest

from _helpers import compare_runs, compare_weights, oracle_step, run_and_check
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
    rng = np.random.default_rng(seed + 1000)
    T = len(rows)
    lengths = lengths_fn(rng, T, B)
    ids_fn = ids_fn or (lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64))
    return synth.make_bag_workload("custom", seed, rows, dims, B, lengths, ids_fn, **kw)


# ---------------------------------------------------------------- the workloads at full size

def test_tiny_pooled_sgd():
    run_and_check(synth.tiny(0))


def test_dlrm_rowwise_adagrad():
    run_and_check(synth.dlrm(0))


def test_mixed_weighted_mean_fp16():
    run_and_check(synth.mixed(0))


def test_mixed_uniform_ids_smaller_batch():
    run_and_check(synth.mixed(1, B=2048, zipf_a=None))


@pytest.mark.parametrize("path", [E.EMB_NOBAG_SORTED, E.EMB_NOBAG_ATOMIC, E.EMB_NOBAG_AUTO])
def test_lm_unpooled_sgd(path):
    run_and_check(synth.lm(0), path=path)


# ---------------------------------------------------------------- variants

@pytest.mark.parametrize("opt", [synth.SGD, synth.ROWWISE_ADAGRAD])
@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.SUM, True),
                                              (synth.MEAN, False), (synth.MEAN, True)])
@pytest.mark.parametrize("wdt", [synth.F32, synth.F16, synth.BF16])
def test_pooled_variants(opt, pooling, weighted, wdt):
    w = custom(3, [300, 50, 2000], [8, 64, 20], 96, lambda r, T, B: r.integers(0, 40, (T, B)),
               optimizer=opt, pooling=pooling, weighted=weighted, weight_dtype=wdt,
               momentum_init=0.5 if opt == synth.ROWWISE_ADAGRAD else 0.0)
    run_and_check(w)


@pytest.mark.parametrize("opt", [synth.SGD, synth.ROWWISE_ADAGRAD])
@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.SUM, True), (synth.MEAN, False),
                                              (synth.MEAN, True)])
def test_repeats_within_bags(opt, pooling, weighted):
    # bags that hit a few rows dozens of times: long runs made of chains of one
    # (row, bag), crossing the 2048-key tiles of the run-length pass
    rows = [50, 3000]
    w = custom(21, rows, [16, 64], 64, lambda r, T, B: r.integers(0, 300, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.7, r.integers(0, 3, n),
                                               r.integers(0, rows[t], n)).astype(np.int64),
               optimizer=opt, pooling=pooling, weighted=weighted, weight_dtype=synth.F16,
               momentum_init=0.5 if opt == synth.ROWWISE_ADAGRAD else 0.0)
    assert w.N > 4 * 2048
    run_and_check(w)


@pytest.mark.parametrize("gdt", [synth.F16, synth.BF16])
def test_half_precision_grad(gdt):
    w = custom(4, [500, 700], [32, 128], 128, lambda r, T, B: r.integers(1, 30, (T, B)),
               grad_dtype=gdt, optimizer=synth.ROWWISE_ADAGRAD)
    run_and_check(w)


@pytest.mark.parametrize("D", [4, 12, 96, 128, 132, 256, 260, 512, 1024])
def test_row_widths_adagrad(D):
    w = custom(5, [64, 33], [D, D], 40, lambda r, T, B: r.integers(0, 50, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    run_and_check(w)


@pytest.mark.parametrize("D", [1028, 2048, 4096])
def test_wide_rows_sgd(D):
    w = custom(6, [40], [D], 30, lambda r, T, B: r.integers(0, 80, (T, B)), optimizer=synth.SGD)
    run_and_check(w)


@pytest.mark.parametrize("D", [1028, 2048, 4096])
@pytest.mark.parametrize("wdt", [synth.F32, synth.F16])
def test_wide_rows_rowwise_adagrad(D, wdt):
    # rows of 2-4 chunks of 1024 (two launches: the state from the chunks' sums of
    # squares, then the update) next to a narrow table of one chunk; hot rows whose
    # runs are long, cut into slices
    w = custom(6, [40, 300], [D, 64], 60, lambda r, T, B: r.integers(0, 80, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD, weight_dtype=wdt, momentum_init=0.5)
    run_and_check(w)


@pytest.mark.parametrize("pooling,weighted", [(synth.MEAN, True), (synth.SUM, True)])
def test_wide_rows_rowwise_adagrad_scaled(pooling, weighted):
    w = custom(23, [500, 70], [2048, 3072], 40, lambda r, T, B: r.integers(0, 30, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD, pooling=pooling, weighted=weighted,
               weight_dtype=synth.BF16, momentum_init=0.25)
    run_and_check(w)


def test_wide_rows_rowwise_adagrad_deterministic():
    # two launches per call, repeated: bitwise the same results run to run, and a
    # second call on the updated weights and state matches two oracle steps
    w = custom(24, [64], [4096], 200, lambda r, T, B: r.integers(0, 40, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    dw1, dw2 = dev.to_device(w), dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        dev.step(plan, dw1)
        dev.step(plan, dw2)
        assert E.emb_plan_status(plan) == E.EMB_OK
        assert np.array_equal(dev.weights_numpy(dw1).view(np.uint32), dev.weights_numpy(dw2).view(np.uint32))
        assert np.array_equal(dw1.momentum.cpu().numpy().view(np.uint32), dw2.momentum.cpu().numpy().view(np.uint32))
        dev.step(plan, dw1)
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)
    ew, em = oracle_step(w)
    w2 = custom(24, [64], [4096], 200, lambda r, T, B: r.integers(0, 40, (T, B)),
                optimizer=synth.ROWWISE_ADAGRAD)
    w2.weights, w2.momentum = ew, em
    ew2, em2 = oracle_step(w2)
    keys = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets)["run_keys"]
    compare_weights(w, dev.weights_numpy(dw1), ew2, keys)
    np.testing.assert_allclose(dw1.momentum.cpu().numpy(), em2, rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("D", [64, 260, 1028, 4096])
@pytest.mark.parametrize("path", [E.EMB_NOBAG_SORTED, E.EMB_NOBAG_ATOMIC])
def test_unpooled_multi_table(D, path):
    w = custom(7, [100, 3000, 17], [D, D, D], 3, lambda r, T, B: r.integers(0, 60, (T, B)),
               nobag=True)
    run_and_check(w, path=path)


# ---------------------------------------------------------------- edge cases

def test_all_lookups_on_one_row():
    # one run of 20000 lookups: several block parts, combined in part order
    w = custom(8, [10, 10], [64, 64], 1000, lambda r, T, B: np.full((T, B), 10),
               ids_fn=lambda r, t, n: np.full(n, 3, np.int64), optimizer=synth.ROWWISE_ADAGRAD)
    run_and_check(w)


def test_hot_rows_many_parts_sgd_fp16():
    w = custom(9, [1000], [128], 4096, lambda r, T, B: r.integers(20, 60, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.5, 0, r.integers(0, 1000, n)).astype(np.int64),
               weight_dtype=synth.F16)
    run_and_check(w)


@pytest.mark.parametrize("L", [31, 32, 33])
def test_run_at_long_threshold(L):
    # every row is hit exactly L times: runs just below / at / above the threshold
    rows = 64
    w = custom(10, [rows], [16], L, lambda r, T, B: np.full((T, B), rows),
               ids_fn=lambda r, t, n: np.tile(np.arange(rows), n // rows).astype(np.int64))
    run_and_check(w)


@pytest.mark.parametrize("thr", [1, 2, 7, 1000])
def test_threshold_values(thr):
    w = custom(11, [200, 100], [16, 32], 64, lambda r, T, B: r.integers(0, 9, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    run_and_check(w, thr=thr)


def test_empty_bags_and_single_table():
    w = custom(12, [5000], [32], 500, lambda r, T, B: r.integers(0, 3, (T, B)) * (r.random((T, B)) < 0.3))
    assert (np.diff(w.offsets) == 0).any()
    run_and_check(w)


def test_zero_lookups_is_a_no_op():
    w = custom(13, [100, 100], [16, 16], 8, lambda r, T, B: np.zeros((T, B), np.int64))
    assert w.N == 0
    dw = dev.to_device(w)
    plan = dev.make_plan(w, max_N=16)
    try:
        dev.step(plan, dw)
        assert E.emb_plan_status(plan) == E.EMB_OK
        assert E.emb_plan_debug_runs(plan, 16)["num_runs"] == 0
    finally:
        E.emb_plan_destroy(plan)
    assert np.array_equal(dev.weights_numpy(dw), w.weights)


def test_tile_boundaries_ragged_tail():
    # sizes around the sort tile (1024) and run-length tile (2048)
    for n in (1023, 1024, 1025, 2047, 2049, 4097):
        w = custom(14 + n, [300], [8], 1, lambda r, T, B, n=n: np.full((T, B), n))
        run_and_check(w)


@pytest.mark.parametrize("rows", [[32], [600], [3000], [300_000], [150_000, 150_000], [(1 << 20) + 5],
                                  [(1 << 24) + 3]])
def test_key_widths(rows):
    # total rows fix the key width: 5 to 25 bits, sorted in 1 to 4 radix passes
    def ids(r, t, n):  # half hot (Zipf), half uniform so that every digit varies
        return np.where(r.random(n) < 0.5, synth.sample_zipf(r, rows[t], 1.05, n), r.integers(0, rows[t], n))

    w = custom(17 + rows[0], rows, [4] * len(rows), 600, lambda r, T, B: r.integers(0, 20, (T, B)), ids_fn=ids)
    run_and_check(w)


def test_large_batch_uses_big_tiles():
    # > 2^21 lookups selects the 4096-lookup sort tiles
    w = custom(15, [50_000, 200_000], [16, 32], 40_000, lambda r, T, B: r.integers(20, 40, (T, B)),
               ids_fn=lambda r, t, n: synth.sample_zipf(r, [50_000, 200_000][t], 1.1, n),
               optimizer=synth.ROWWISE_ADAGRAD)
    assert w.N > (1 << 21)
    run_and_check(w)


def test_custom_momentum_offsets_and_max_sizes():
    w = custom(16, [100, 200], [16, 16], 32, lambda r, T, B: r.integers(0, 10, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    w.momentum_offsets = np.array([200, 0], np.int64)  # table 1's state first
    w.momentum = np.random.default_rng(0).uniform(0, 1, 300).astype(np.float32)
    run_and_check(w, plan_kw=dict(max_N=w.N * 3 + 7, max_B=w.B + 5))


def test_repeated_calls_on_one_plan_deterministic():
    w = synth.dlrm(1)
    dw1, dw2 = dev.to_device(w), dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        dev.step(plan, dw1)
        dev.step(plan, dw2)
        assert E.emb_plan_status(plan) == E.EMB_OK
        # bitwise run-to-run reproducible
        assert np.array_equal(dev.weights_numpy(dw1).view(np.uint32), dev.weights_numpy(dw2).view(np.uint32))
        assert np.array_equal(dw1.momentum.cpu().numpy().view(np.uint32), dw2.momentum.cpu().numpy().view(np.uint32))
        # a second step on the same weights matches two oracle steps
        dev.step(plan, dw1)
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)
    ew, em = oracle_step(w)
    w2 = synth.dlrm(1)
    w2.weights, w2.momentum = ew, em
    ew2, em2 = oracle_step(w2)
    keys = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets)["run_keys"]
    compare_weights(w, dev.weights_numpy(dw1), ew2, keys)
    np.testing.assert_allclose(dw1.momentum.cpu().numpy(), em2, rtol=1e-4, atol=1e-5)


# ---------------------------------------------------------------- device-detected errors

def _expect_status(w, status, path=E.EMB_NOBAG_AUTO, flags=0):
    dw = dev.to_device(w)
    w0 = dev.weights_numpy(dw).copy()
    m0 = None if dw.momentum is None else dw.momentum.cpu().numpy().copy()
    plan = dev.make_plan(w, flags=flags)
    try:
        dev.step(plan, dw, path=path)
        assert E.emb_plan_status(plan) == status
        assert E.emb_plan_status(plan) == E.EMB_OK  # the latched error was cleared
    finally:
        E.emb_plan_destroy(plan)
    assert np.array_equal(dev.weights_numpy(dw), w0), "weights modified despite the error"
    if m0 is not None:
        assert np.array_equal(dw.momentum.cpu().numpy(), m0)


# both fronts of the sorted path: the small-batch one (a cluster per table) and the multi-block one
FRONTS = [0, E.EMB_FLAG_NO_CLUSTER_FRONT]


@pytest.mark.parametrize("bad", [-1, 100, 1 << 40])
@pytest.mark.parametrize("path", [E.EMB_NOBAG_SORTED, E.EMB_NOBAG_ATOMIC, None])
@pytest.mark.parametrize("front", FRONTS)
def test_index_out_of_range_leaves_weights(bad, path, front):
    w = custom(17, [100, 50], [16, 16], 64, lambda r, T, B: r.integers(1, 5, (T, B)),
               nobag=path is not None, optimizer=synth.SGD)
    w.indices[w.N // 2] = bad
    _expect_status(w, E.EMB_ERR_INDEX_OUT_OF_RANGE, path=path or E.EMB_NOBAG_AUTO, flags=front)


@pytest.mark.parametrize("front", FRONTS)
def test_malformed_offsets_detected(front):
    w = custom(18, [100, 50], [16, 16], 64, lambda r, T, B: r.integers(1, 5, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    w.offsets = w.offsets.copy()
    w.offsets[10], w.offsets[11] = w.offsets[11], w.offsets[10] - 1  # decreasing
    _expect_status(w, E.EMB_ERR_INVALID_ARG, flags=front)


@pytest.mark.parametrize("front", FRONTS)
def test_malformed_table_bounds_detected(front):
    # the first table's lookups claimed to end past the batch: every segment is
    # clamped into the batch, nothing is read or written out of bounds
    w = custom(22, [100, 50], [16, 16], 64, lambda r, T, B: r.integers(1, 5, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    w.offsets = w.offsets.copy()
    w.offsets[w.B] = w.N + 1000
    _expect_status(w, E.EMB_ERR_INVALID_ARG, flags=front)


@pytest.mark.parametrize("front", FRONTS)
def test_forced_lookback_timeout_is_reported_not_hung(front):
    # many sort tiles, so some block must wait on another; the test flag makes
    # every such wait give up at once
    w = custom(19, [5000], [16], 2000, lambda r, T, B: r.integers(1, 8, (T, B)),
               optimizer=synth.ROWWISE_ADAGRAD)
    assert w.N > 4 * 1024
    _expect_status(w, E.EMB_ERR_TIMEOUT, flags=E.EMB_FLAG_DEBUG_FORCE_TIMEOUT | front)


def test_call_argument_errors():
    w = custom(20, [100], [16], 8, lambda r, T, B: r.integers(1, 5, (T, B)))
    dw = dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        with pytest.raises(E.EmbError) as e:
            E.emb_bag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, w.N + 1, w.B, None,
                              dw.grad_output, 0, 0.1)  # N above max_N
        assert e.value.status == E.EMB_ERR_INVALID_ARG
        with pytest.raises(E.EmbError) as e:
            E.emb_bag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B + 1, None,
                              dw.grad_output, 0, 0.1)  # B above max_B
        assert e.value.status == E.EMB_ERR_INVALID_ARG
        with pytest.raises(E.EmbError) as e:
            E.emb_bag_bwd_sgd(plan, dw.weights.data_ptr() + 4, dw.indices, dw.offsets, w.N, w.B,
                              None, dw.grad_output, 0, 0.1)  # misaligned weights
        assert e.value.status == E.EMB_ERR_INVALID_ARG
        with pytest.raises(E.EmbError) as e:
            E.emb_bag_bwd_rowwise_adagrad(plan, dw.weights, None, dw.indices, dw.offsets, w.N,
                                          w.B, None, dw.grad_output, 0, 0.1, 1e-8)  # no momentum
        assert e.value.status == E.EMB_ERR_INVALID_ARG
        with pytest.raises(E.EmbError) as e:
            E.emb_bag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B, None,
                              dw.grad_output, 7, 0.1)  # bad pooling mode
        assert e.value.status == E.EMB_ERR_INVALID_ARG
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)


def test_atomic_path_needs_fp32_weights():
    w = custom(21, [100], [16], 8, lambda r, T, B: r.integers(1, 5, (T, B)), nobag=True,
               weight_dtype=synth.F16)
    dw = dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        with pytest.raises(E.EmbError) as e:
            dev.step(plan, dw, path=E.EMB_NOBAG_ATOMIC)
        assert e.value.status == E.EMB_ERR_UNSUPPORTED
        dev.step(plan, dw, path=E.EMB_NOBAG_AUTO)  # falls to the sorted path
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)


def test_profiling_stage_times():
    w = synth.dlrm(2)
    dw = dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        E.emb_plan_set_profiling(plan, True)
        dev.step(plan, dw)
        ms = E.emb_plan_stage_ms(plan)
        assert ms.shape == (5,) and np.all(ms >= 0) and ms.sum() > 0
    finally:
        E.emb_plan_destroy(plan)
