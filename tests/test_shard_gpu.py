"""GPU parity of the row-sharded exchange: bucketize and merge through the C ABI
against the oracle (bit for bit: integer work and one fp32 division per scale),
and a W-rank sharded step emulated on one GPU (every rank's bucketize, the
all-to-all as device copies, every owner's merge and backward on its own plan)
against the unsharded oracle step on the global batch.
"""
import numpy as np
import pytest

from _helpers import ATOL, RTOL
import oracle
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import shard as S
from sparse_embedding_bag_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_embedding_bag_gb300 import build
    build.build()
    E.load()


def batch(seed, rows, dims, B, max_len=12, weighted=False, empty_share=0.0, **kw):
    rng = np.random.default_rng(seed + 5000)
    lengths = rng.integers(0, max_len, (len(rows), B)) * (rng.random((len(rows), B)) >= empty_share)
    return synth.make_bag_workload("shg", seed, rows, dims, B, lengths,
                                   lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                   weighted=weighted, **kw)


def gpu_bucketize(sh, w, W, mean, scales=True):
    import torch
    BT = w.T * w.B
    idx = torch.from_numpy(w.indices).cuda()
    off = torch.from_numpy(w.offsets).cuda()
    psw = None if w.per_sample_weights is None else torch.from_numpy(w.per_sample_weights).cuda()
    so = torch.full((W, BT + 1), -7, dtype=torch.int64, device="cuda")
    si = torch.full((max(w.N, 1),), -7, dtype=torch.int64, device="cuda")
    ss = torch.full((max(w.N, 1),), -7.0, dtype=torch.float32, device="cuda") if scales else None
    counts = E.emb_shard_bucketize(sh, idx, off, w.N, w.B, psw, E.EMB_POOL_MEAN if mean else E.EMB_POOL_SUM,
                                   so, si, ss)
    return so.cpu().numpy(), si.cpu().numpy()[:w.N], None if ss is None else ss.cpu().numpy()[:w.N], counts


@pytest.mark.parametrize("W,mode", [(1, "sum"), (8, "sum"), (8, "weighted"), (8, "mean"),
                                    (3, "weighted_mean"), (64, "sum"), (8, "cyclic_weighted_mean"),
                                    (5, "cyclic_sum"), (256, "cyclic_sum")])
def test_bucketize_parity(W, mode):
    rows = [5000, 300, 70, 1]
    w = batch(1, rows, [16, 8, 4, 4], 256, weighted="weighted" in mode, empty_share=0.2)
    mean, cyclic = "mean" in mode, "cyclic" in mode
    rb = S.even_row_bounds(rows, W)  # the one-row table leaves W-1 ranks no rows
    sh = E.emb_shard_create_cyclic(0, w.T, W, rows, w.B) if cyclic else E.emb_shard_create(0, w.T, W, rb, w.B)
    try:
        so, si, ss, sc = gpu_bucketize(sh, w, W, mean)
    finally:
        E.emb_shard_destroy(sh)
    eo, ei, es, ec = oracle.bucketize(w.T, w.B, rb, w.indices, w.offsets,
                                      per_sample_weights=w.per_sample_weights, mean=mean, cyclic=cyclic)
    assert np.array_equal(sc, ec)
    assert np.array_equal(so, eo)
    assert np.array_equal(si, ei)
    assert np.array_equal(ss.view(np.uint32), es.view(np.uint32))


def test_bucketize_uneven_ranges_and_no_scales():
    rows = [60, 9, 33]
    w = batch(2, rows, [4, 4, 8], 40, max_len=9)
    rb = np.array([[0, 20, 59, 60], [0, 9, 9, 9], [0, 1, 17, 33]], np.int64)
    sh = E.emb_shard_create(0, 3, 3, rb, 64)  # max_B above B
    try:
        so, si, ss, sc = gpu_bucketize(sh, w, 3, False, scales=False)
        # a second call on the same map gives the same result
        so2, si2, _, sc2 = gpu_bucketize(sh, w, 3, False, scales=False)
    finally:
        E.emb_shard_destroy(sh)
    eo, ei, _, ec = oracle.bucketize(w.T, w.B, rb, w.indices, w.offsets)
    assert np.array_equal(so, eo) and np.array_equal(si, ei) and np.array_equal(sc, ec)
    assert np.array_equal(so2, eo) and np.array_equal(si2, ei) and np.array_equal(sc2, ec)


def test_bucketize_no_lookups():
    w = batch(3, [100, 100], [16, 16], 8, empty_share=1.0)
    assert w.N == 0
    sh = E.emb_shard_create(0, 2, 4, S.even_row_bounds([100, 100], 4), 8)
    try:
        so, _, _, sc = gpu_bucketize(sh, w, 4, False)
    finally:
        E.emb_shard_destroy(sh)
    assert np.all(so == 0) and np.all(sc == 0)


def test_bucketize_reports_bad_index():
    w = batch(4, [100, 50], [16, 16], 20, max_len=5)
    w.indices[-1] = 50  # one past the end of table 1
    sh = E.emb_shard_create(0, 2, 2, S.even_row_bounds([100, 50], 2), 20)
    try:
        with pytest.raises(E.EmbError) as ei:
            gpu_bucketize(sh, w, 2, False)
        assert ei.value.status == E.EMB_ERR_INDEX_OUT_OF_RANGE
        w.indices[-1] = 49
        gpu_bucketize(sh, w, 2, False)  # the error was cleared
    finally:
        E.emb_shard_destroy(sh)


def exchange_np(parts, W):
    """Owner r's received parts: (offsets [W, BT+1], indices, scales) in source order."""
    out = []
    for r in range(W):
        offs, idx, sc = [], [], []
        for so, si, ss, cnt in parts:
            a = int(cnt[:r].sum())
            offs.append(so[r])
            idx.append(si[a:a + cnt[r]])
            sc.append(ss[a:a + cnt[r]])
        out.append((np.stack(offs), np.concatenate(idx), np.concatenate(sc)))
    return out


@pytest.mark.parametrize("W", [2, 5])
def test_merge_parity(W):
    import torch
    rows = [800, 60, 300]
    T, B = 3, 33
    sources = [batch(10 + s, rows, [8, 4, 16], B, weighted=True, empty_share=0.1) for s in range(W)]
    rb = S.even_row_bounds(rows, W)
    parts = [oracle.bucketize(T, B, rb, s.indices, s.offsets, per_sample_weights=s.per_sample_weights,
                              mean=True) for s in sources]
    sh = E.emb_shard_create(0, T, W, rb, B)
    try:
        for r, (ro, ri, rs) in enumerate(exchange_np(parts, W)):
            n = ri.size
            mo = torch.full((T * W * B + 1,), -3, dtype=torch.int64, device="cuda")
            mi = torch.full((max(n, 1),), -3, dtype=torch.int64, device="cuda")
            ms = torch.full((max(n, 1),), -3.0, dtype=torch.float32, device="cuda")
            E.emb_shard_merge(sh, torch.from_numpy(ro).cuda(), torch.from_numpy(ri).cuda(),
                              torch.from_numpy(rs).cuda(), n, B, mo, mi, ms)
            assert E.emb_shard_status(sh) == E.EMB_OK
            eo, ei, es = oracle.merge(T, B, W, ro, ri, rs)
            assert np.array_equal(mo.cpu().numpy(), eo)
            assert np.array_equal(mi.cpu().numpy()[:n], ei)
            assert np.array_equal(ms.cpu().numpy()[:n].view(np.uint32), es.view(np.uint32))
    finally:
        E.emb_shard_destroy(sh)


def test_merge_reports_inconsistent_offsets():
    import torch
    rows, T, B, W = [100, 40], 2, 10, 2
    sources = [batch(20 + s, rows, [4, 4], B) for s in range(W)]
    rb = S.even_row_bounds(rows, W)
    parts = [oracle.bucketize(T, B, rb, s.indices, s.offsets) for s in sources]
    ro, ri, rs = exchange_np(parts, W)[0]
    ro = ro.copy()
    ro[0, -1] += 5  # source 0 claims five lookups more than were received
    n = ri.size
    sh = E.emb_shard_create(0, T, W, rb, B)
    try:
        mo = torch.zeros(T * W * B + 1, dtype=torch.int64, device="cuda")
        mi = torch.zeros(max(n, 1), dtype=torch.int64, device="cuda")
        E.emb_shard_merge(sh, torch.from_numpy(ro).cuda(), torch.from_numpy(ri).cuda(), None, n, B, mo, mi, None)
        assert E.emb_shard_status(sh) == E.EMB_ERR_INVALID_ARG
    finally:
        E.emb_shard_destroy(sh)


def emulated_step(rows, dims, B, W, optimizer, weighted, mean, seed=30, cyclic=False):
    """W ranks on one GPU: every rank's bucketize, the all-to-all as device copies,
    every owner's merge, backward (and forward) on its own plan. Returns the
    unsharded weights, state and every rank's forward output."""
    import torch
    T = len(rows)
    model = synth.make_bag_workload("shm", seed, rows, dims, B, np.ones((T, B), np.int64),
                                    lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                    optimizer=optimizer, momentum_init=0.5, lr=0.05)
    sources = [batch(seed + 1 + s, rows, dims, B, weighted=weighted, empty_share=0.1) for s in range(W)]
    rb = S.even_row_bounds(rows, W)
    need_scales = weighted or mean
    sends = []
    for s, src in enumerate(sources):
        sh = E.emb_shard_create_cyclic(0, T, W, rows, B) if cyclic else E.emb_shard_create(0, T, W, rb, B)
        try:
            so = torch.empty((W, T * B + 1), dtype=torch.int64, device="cuda")
            si = torch.empty(max(src.N, 1), dtype=torch.int64, device="cuda")
            ss = torch.empty(max(src.N, 1), dtype=torch.float32, device="cuda") if need_scales else None
            psw = None if src.per_sample_weights is None else torch.from_numpy(src.per_sample_weights).cuda()
            cnt = E.emb_shard_bucketize(sh, torch.from_numpy(src.indices).cuda(),
                                        torch.from_numpy(src.offsets).cuda(), src.N, B, psw,
                                        E.EMB_POOL_MEAN if mean else E.EMB_POOL_SUM, so, si, ss)
        finally:
            E.emb_shard_destroy(sh)
        sends.append((so, si, ss, cnt))
    grad = torch.from_numpy(np.concatenate([s.grad_output for s in sources])).cuda()
    weights_full = np.array(model.weights, copy=True)
    mom_full = None if model.momentum is None else model.momentum.copy()
    fwd = np.zeros((W * B, int(np.sum(dims))), np.float64)
    for r in range(W):
        # the all-to-all: owner r's part of every source, in source order
        ro = torch.stack([so[r] for so, _, _, _ in sends])
        pieces = [(si[int(c[:r].sum()):int(c[:r].sum()) + int(c[r])],
                   None if ss is None else ss[int(c[:r].sum()):int(c[:r].sum()) + int(c[r])])
                  for _, si, ss, c in sends]
        ri = torch.cat([p[0] for p in pieces])
        rs = torch.cat([p[1] for p in pieces]) if need_scales else None
        n = int(ri.numel())
        local, hsc, Do, wo = S.local_tables(rows, dims, rb, r, W, cyclic)
        own = S.owned_rows(rows, rb, r, W, cyclic)
        sh = E.emb_shard_create(0, T, W, rb, B)  # merge does not depend on the map
        plan = E.emb_bwd_plan(0, T, hsc, Do, wo, None, synth.F32, synth.F32, max(n, 1), W * B, 0, 0)
        try:
            mo = torch.empty(T * W * B + 1, dtype=torch.int64, device="cuda")
            mi = torch.empty(max(n, 1), dtype=torch.int64, device="cuda")
            ms = torch.empty(max(n, 1), dtype=torch.float32, device="cuda") if need_scales else None
            E.emb_shard_merge(sh, ro, ri if n else mi, rs if (n or not need_scales) else ms, n, B, mo, mi, ms)
            assert E.emb_shard_status(sh) == E.EMB_OK
            gidx = [(model.weights_offsets[t] + own[t][:, None] * dims[t] + np.arange(dims[t])).reshape(-1)
                    for t in range(T)]
            wl = torch.from_numpy(np.concatenate([model.weights[g] for g in gidx])).cuda()
            ml = None if mom_full is None else torch.from_numpy(np.concatenate(
                [model.momentum[model.hash_size_cumsum[t] + own[t]] for t in range(T)])).cuda()
            out = torch.zeros((W * B, int(np.sum(dims))), dtype=torch.float32, device="cuda")
            if n:
                E.emb_bag_fwd(plan, wl, mi, mo, n, W * B, ms, E.EMB_POOL_SUM, out, 0)
                if optimizer == synth.SGD:
                    E.emb_bag_bwd_sgd(plan, wl, mi, mo, n, W * B, ms, grad, E.EMB_POOL_SUM, model.lr)
                else:
                    E.emb_bag_bwd_rowwise_adagrad(plan, wl, ml, mi, mo, n, W * B, ms, grad,
                                                  E.EMB_POOL_SUM, model.lr, model.eps)
                assert E.emb_plan_status(plan) == E.EMB_OK
            fwd += out.cpu().numpy()  # the reduce-scatter's sum over owners
            wl_np = wl.cpu().numpy()
            for t in range(T):
                D = int(dims[t])
                weights_full[gidx[t]] = wl_np[wo[t]:wo[t] + own[t].size * D]
                if ml is not None:
                    mom_full[model.hash_size_cumsum[t] + own[t]] = ml.cpu().numpy()[hsc[t]:hsc[t + 1]]
        finally:
            E.emb_plan_destroy(plan)
            E.emb_shard_destroy(sh)
    return model, sources, weights_full, mom_full, fwd


@pytest.mark.parametrize("optimizer,weighted,mean,cyclic", [(synth.SGD, False, False, False),
                                                            (synth.SGD, True, True, False),
                                                            (synth.ROWWISE_ADAGRAD, True, False, False),
                                                            (synth.SGD, False, False, True),
                                                            (synth.ROWWISE_ADAGRAD, True, True, True)])
def test_emulated_sharded_step_equals_unsharded(optimizer, weighted, mean, cyclic):
    rows, dims, B, W = [3000, 200, 57], [32, 8, 64], 128, 4
    model, sources, got_w, got_m, fwd = emulated_step(rows, dims, B, W, optimizer, weighted, mean,
                                                      cyclic=cyclic)
    T = len(rows)
    # the unsharded step on the global batch (bag (t, s*B + b) = source s's bag (t, b))
    gidx, goff, gpsw = [], [0], []
    for t in range(T):
        for s in sources:
            for b in range(B):
                a, e = int(s.offsets[t * B + b]), int(s.offsets[t * B + b + 1])
                gidx.extend(s.indices[a:e].tolist())
                if s.per_sample_weights is not None:
                    gpsw.extend(s.per_sample_weights[a:e].tolist())
                goff.append(len(gidx))
    grad = np.concatenate([s.grad_output for s in sources])
    ref_w = np.array(model.weights, copy=True)
    ref_m = None if model.momentum is None else model.momentum.copy()
    oracle.backward(T, W * B, model.hash_size_cumsum, model.D_offsets, model.weights_offsets, ref_w,
                    np.array(gidx, np.int64), np.array(goff, np.int64), grad, optimizer=optimizer,
                    lr=model.lr, eps=model.eps, momentum=ref_m,
                    per_sample_weights=np.array(gpsw, np.float32) if gpsw else None, mean=mean)
    np.testing.assert_allclose(got_w, ref_w, rtol=RTOL, atol=ATOL)
    untouched = ref_w == model.weights
    assert np.array_equal(got_w[untouched], model.weights[untouched])
    if ref_m is not None:
        np.testing.assert_allclose(got_m, ref_m, rtol=RTOL, atol=ATOL)
    # forward: every rank's own bags, from the owners' partial sums
    for s, src in enumerate(sources):
        ref = oracle.forward(T, B, model.hash_size_cumsum, model.D_offsets, model.weights_offsets,
                             model.weights, src.indices, src.offsets,
                             per_sample_weights=src.per_sample_weights, mean=mean)
        np.testing.assert_allclose(fwd[s * B:(s + 1) * B], ref, rtol=RTOL, atol=ATOL)
