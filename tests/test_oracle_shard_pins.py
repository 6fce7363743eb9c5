"""Pins for the oracle's row-sharded exchange (bucketize on every source rank,
merge on every owner) against things other than itself.

* one rank: bucketizing is the identity on offsets and indices, and the scales
  are the per-sample weights, or numpy's fp32 quotient psw / L under mean pooling;
* several ranks with uneven and empty ranges: brute force per bag (a Python
  filter of each bag's lookups by range), counts summing to N, rows relative to
  the owner's range;
* merge: equals the table-major CSR of all sources' batches side by side, built
  by brute force from the sources' own batches;
* composition: bucketize on every source, all-to-all, merge and the oracle's
  backward on every owner's shard equals the unsharded backward of the global
  batch (bit for bit with unweighted sum pooling, whose summation order is the
  same; within fp32 rounding of the scale under mean / weighted pooling), for
  SGD and row-wise Adagrad. A wrong owner, a dropped lookup, the shard's instead
  of the whole bag's length for the mean, or a wrong bag order fails it.
"""
import numpy as np
import pytest

from sparse_embedding_bag_gb300 import synth


def even_bounds(rows, W):
    return np.array([[r * k // W for k in range(W + 1)] for r in rows], np.int64)


def batch(seed, rows, dims, B, max_len=6, weighted=False, weight_dtype=synth.F32, **kw):
    rng = np.random.default_rng(seed)
    return synth.make_bag_workload("sh", seed, rows, dims, B, rng.integers(0, max_len, (len(rows), B)),
                                   lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                   weighted=weighted, weight_dtype=weight_dtype, **kw)


@pytest.mark.parametrize("mode", ["sum", "weighted", "mean", "weighted_mean"])
def test_one_rank_is_identity(oracle_mod, mode):
    w = batch(1, [50, 7], [8, 4], 20, weighted="weighted" in mode)
    mean = "mean" in mode
    rb = even_bounds(w.rows, 1)
    so, si, ss, sc = oracle_mod.bucketize(w.T, w.B, rb, w.indices, w.offsets,
                                          per_sample_weights=w.per_sample_weights, mean=mean)
    assert np.array_equal(so[0], w.offsets) and np.array_equal(si, w.indices)
    assert sc.tolist() == [w.N]
    psw = w.per_sample_weights if w.per_sample_weights is not None else np.ones(w.N, np.float32)
    L = np.repeat(np.diff(w.offsets), np.diff(w.offsets)).astype(np.float32)
    exp = (psw / L).astype(np.float32) if mean else psw
    assert np.array_equal(ss.view(np.uint32), exp.astype(np.float32).view(np.uint32))


def test_brute_force_uneven_ranges(oracle_mod):
    rows = [60, 9, 33]
    w = batch(2, rows, [4, 4, 8], 15, max_len=9, weighted=True)
    # rank 1 owns nothing of table 1; rank 2 owns a single row of table 0
    rb = np.array([[0, 20, 59, 60], [0, 9, 9, 9], [0, 1, 17, 33]], np.int64)
    so, si, ss, sc = oracle_mod.bucketize(w.T, w.B, rb, w.indices, w.offsets,
                                          per_sample_weights=w.per_sample_weights)
    W = 3
    assert sc.sum() == w.N and so.shape == (W, w.T * w.B + 1)
    start = np.concatenate([[0], np.cumsum(sc)])
    for r in range(W):
        assert so[r, 0] == 0 and so[r, -1] == sc[r]
        for bt in range(w.T * w.B):
            t = bt // w.B
            want = [(int(w.indices[i]) - rb[t, r], w.per_sample_weights[i])
                    for i in range(w.offsets[bt], w.offsets[bt + 1])
                    if rb[t, r] <= w.indices[i] < rb[t, r + 1]]
            a, b = start[r] + so[r, bt], start[r] + so[r, bt + 1]
            got = list(zip(si[a:b].tolist(), ss[a:b].tolist()))
            assert got == [(i, float(s)) for i, s in want]
            assert all(0 <= i < rb[t, r + 1] - rb[t, r] for i, _ in got)


def cyclic_bounds(rows, W):
    """The row counts in the last column (all a cyclic map reads)."""
    rb = np.zeros((len(rows), W + 1), np.int64)
    rb[:, W] = rows
    return rb


@pytest.mark.parametrize("W", [1, 4])
def test_cyclic_brute_force(oracle_mod, W):
    rows = [60, 3, 33]  # table 1 has fewer rows than ranks: rank 3 owns none of it
    w = batch(4, rows, [4, 4, 8], 15, max_len=9, weighted=True)
    so, si, ss, sc = oracle_mod.bucketize(w.T, w.B, cyclic_bounds(rows, W), w.indices, w.offsets,
                                          per_sample_weights=w.per_sample_weights, cyclic=True)
    assert sc.sum() == w.N
    start = np.concatenate([[0], np.cumsum(sc)])
    for r in range(W):
        for bt in range(w.T * w.B):
            want = [(int(w.indices[i]) // W, w.per_sample_weights[i])
                    for i in range(w.offsets[bt], w.offsets[bt + 1]) if int(w.indices[i]) % W == r]
            a, b = start[r] + so[r, bt], start[r] + so[r, bt + 1]
            assert list(zip(si[a:b].tolist(), ss[a:b].tolist())) == [(i, float(s)) for i, s in want]
    if W == 1:
        assert np.array_equal(si, w.indices) and np.array_equal(so[0], w.offsets)


def test_out_of_range_index_is_an_error(oracle_mod):
    w = batch(3, [10, 10], [4, 4], 4, max_len=3)
    w.indices[-1] = 10
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.bucketize(w.T, w.B, even_bounds(w.rows, 2), w.indices, w.offsets)


def exchange(oracle_mod, sources, rb, mean, cyclic=False):
    """Bucketize every source's batch and deliver owner r's parts, in source order."""
    parts = [oracle_mod.bucketize(src.T, src.B, rb, src.indices, src.offsets,
                                  per_sample_weights=src.per_sample_weights, mean=mean, cyclic=cyclic)
             for src in sources]
    W = rb.shape[1] - 1
    recv = []
    for r in range(W):
        offs, idx, sc = [], [], []
        for so, si, ss, cnt in parts:
            a = int(cnt[:r].sum())
            offs.append(so[r])
            idx.append(si[a:a + cnt[r]])
            sc.append(ss[a:a + cnt[r]])
        recv.append((np.stack(offs), np.concatenate(idx), np.concatenate(sc)))
    return recv


def global_batch(sources):
    """All sources' batches side by side: bag (t, s*B + b) = source s's bag (t, b)."""
    T, B, W = sources[0].T, sources[0].B, len(sources)
    idx, off, psw = [], [0], []
    for t in range(T):
        for s in sources:
            for b in range(B):
                bt = t * B + b
                a, e = int(s.offsets[bt]), int(s.offsets[bt + 1])
                idx.extend(s.indices[a:e].tolist())
                if s.per_sample_weights is not None:
                    psw.extend(s.per_sample_weights[a:e].tolist())
                off.append(len(idx))
    grad = np.concatenate([s.grad_output for s in sources])
    return (np.array(idx, np.int64), np.array(off, np.int64),
            np.array(psw, np.float32) if psw else None, grad, W * B)


def test_merge_equals_global_batch_by_brute_force(oracle_mod):
    rows = [40, 12]
    sources = [batch(10 + s, rows, [4, 8], 6, max_len=5) for s in range(3)]
    rb = even_bounds(rows, 3)
    recv = exchange(oracle_mod, sources, rb, mean=False)
    gidx, goff, _, _, GB = global_batch(sources)
    for r, (ro, ri, rs) in enumerate(recv):
        mo, mi, ms = oracle_mod.merge(2, 6, 3, ro, ri, rs)
        # brute force: the global batch's lookups of r's rows, relative to r's range
        want_idx, want_off = [], [0]
        for q in range(2 * GB):
            t = q // GB
            for i in range(goff[q], goff[q + 1]):
                if rb[t, r] <= gidx[i] < rb[t, r + 1]:
                    want_idx.append(int(gidx[i]) - rb[t, r])
            want_off.append(len(want_idx))
        assert mo.tolist() == want_off and mi.tolist() == want_idx
        assert np.all(ms == 1.0)


def owned_rows(w, rb, r, cyclic):
    """Rows of every table that owner r holds, in its local order."""
    W = rb.shape[1] - 1
    if cyclic:
        return [np.arange(r, int(w.rows[t]), W) for t in range(w.T)]
    return [np.arange(rb[t, r], rb[t, r + 1]) for t in range(w.T)]


def shard_layout(w, rb, r, cyclic=False):
    """Owner r's tables: its rows of every table (hash_size_cumsum, weights
    offsets, weights and row-wise state gathered from the full arrays)."""
    own = owned_rows(w, rb, r, cyclic)
    local = np.array([o.size for o in own], np.int64)
    hsc = np.concatenate([[0], np.cumsum(local)]).astype(np.int64)
    wo = np.concatenate([[0], np.cumsum(local * w.dims)[:-1]]).astype(np.int64)
    weights = np.concatenate([w.weights[(w.weights_offsets[t] + own[t][:, None] * w.dims[t] +
                                         np.arange(w.dims[t])).reshape(-1)] for t in range(w.T)])
    mom = None if w.momentum is None else np.concatenate(
        [w.momentum[w.hash_size_cumsum[t] + own[t]] for t in range(w.T)])
    return hsc, wo, weights.copy(), mom


def unshard(w, rb, shards, cyclic=False):
    """Full weights (and state) from the owners' rows."""
    weights, mom = np.array(w.weights, copy=True), None if w.momentum is None else w.momentum.copy()
    for r, (sw, sm) in enumerate(shards):
        hsc, wo, _, _ = shard_layout(w, rb, r, cyclic)
        own = owned_rows(w, rb, r, cyclic)
        for t in range(w.T):
            D = int(w.dims[t])
            dst = (w.weights_offsets[t] + own[t][:, None] * D + np.arange(D)).reshape(-1)
            weights[dst] = sw[wo[t]:wo[t] + own[t].size * D]
            if mom is not None:
                mom[w.hash_size_cumsum[t] + own[t]] = sm[hsc[t]:hsc[t + 1]]
    return weights, mom


@pytest.mark.parametrize("opt,weighted,mean,cyclic", [(synth.SGD, False, False, False),
                                                      (synth.SGD, True, True, False),
                                                      (synth.ROWWISE_ADAGRAD, False, False, False),
                                                      (synth.ROWWISE_ADAGRAD, True, False, False),
                                                      (synth.SGD, False, True, False),
                                                      (synth.SGD, False, False, True),
                                                      (synth.ROWWISE_ADAGRAD, True, True, True)])
def test_sharded_step_equals_unsharded(oracle_mod, opt, weighted, mean, cyclic):
    rows, dims, B, W = [70, 25, 300], [8, 4, 16], 12, 3
    sources = [batch(20 + s, rows, dims, B, max_len=8, weighted=weighted, optimizer=opt)
               for s in range(W)]
    w = sources[0]  # the model (weights, state) is the same on every source
    rb = cyclic_bounds(rows, W) if cyclic else even_bounds(rows, W)
    if not cyclic:
        rb[1] = [0, 3, 4, 25]  # uneven: an owner with one row of table 1
    recv = exchange(oracle_mod, sources, rb, mean, cyclic)
    gidx, goff, gpsw, grad, GB = global_batch(sources)
    shards = []
    for r in range(W):
        mo, mi, ms = oracle_mod.merge(w.T, B, W, *recv[r])
        hsc, wo, weights, mom = shard_layout(w, rb, r, cyclic)
        if mi.size:
            oracle_mod.backward(w.T, GB, hsc, w.D_offsets, wo, weights, mi, mo, grad,
                                optimizer=opt, lr=w.lr, eps=w.eps, momentum=mom,
                                per_sample_weights=None if not (weighted or mean) else ms)
        shards.append((weights, mom))
    got_w, got_m = unshard(w, rb, shards, cyclic)
    ref_w = np.array(w.weights, copy=True)
    ref_m = None if w.momentum is None else w.momentum.copy()
    oracle_mod.backward(w.T, GB, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, ref_w, gidx,
                        goff, grad, optimizer=opt, lr=w.lr, eps=w.eps, momentum=ref_m,
                        per_sample_weights=gpsw, mean=mean)
    assert not np.array_equal(ref_w, w.weights)
    if weighted or mean:
        np.testing.assert_allclose(got_w, ref_w, rtol=1e-6, atol=1e-7)
        if ref_m is not None:
            np.testing.assert_allclose(got_m, ref_m, rtol=1e-6, atol=1e-9)
    else:
        assert np.array_equal(got_w.view(np.uint32), ref_w.view(np.uint32))
        if ref_m is not None:
            assert np.array_equal(got_m.view(np.uint32), ref_m.view(np.uint32))
