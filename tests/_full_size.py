"""Sampled-row parity at full size: the step runs whole on the device; the
oracle recomputes sampled rows one by one, each as a one-row problem built from
every lookup of that row (its gradient rows and the row's old state). Rows of a
linear index are independent under the per-row optimizers, so each sampled row
of the full step must equal its one-row problem: fp16 / bf16 weights within one
ulp, or within the derived bound of the device's fp32 arithmetic where an update
cancels (tests/_bounds.py)."""
import numpy as np

import oracle
from _bounds import check16
from sparse_embedding_bag_gb300 import synth


def sampled_rows_check(w, step, hot_per_table=4, n_random=48, n_untouched=8, seed=0):
    """w: a pooled, unweighted, sum-pooled row-wise Adagrad workload whose arrays
    are torch tensors (any device); step(): runs the full step in place on them.
    Returns the number of sampled rows checked."""
    import torch
    dev = w.indices.device
    T, B, D = w.T, w.B, int(w.dims[0])
    assert np.all(w.dims == D) and w.pooling == synth.SUM and w.per_sample_weights is None
    assert w.optimizer == synth.ROWWISE_ADAGRAD and w.momentum_offsets is None
    hsc = torch.as_tensor(w.hash_size_cumsum, device=dev)
    wo = torch.as_tensor(w.weights_offsets, device=dev)
    lengths = w.offsets[1:] - w.offsets[:-1]
    bag = torch.repeat_interleave(torch.arange(T * B, device=dev), lengths)
    t_of = bag // B
    keys = hsc[t_of] + w.indices
    uniq = torch.unique(keys)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    # the hottest rows (ids are Zipf-ranked: row r has rank r + 1) of the first and
    # last table, random touched rows, and random rows no lookup hits
    hot = torch.tensor([int(w.hash_size_cumsum[t]) + r for t in (0, T - 1) for r in range(hot_per_table)],
                       device=dev)
    touched = uniq[torch.randint(0, uniq.numel(), (n_random,), generator=gen).to(dev)]
    cand = torch.randint(0, int(w.hash_size_cumsum[-1]), (64 * n_untouched,), generator=gen).to(dev)
    untouched = cand[~torch.isin(cand, uniq)][:n_untouched]
    sample = torch.unique(torch.cat([hot, touched, untouched]))
    t_s = torch.searchsorted(hsc, sample, right=True) - 1
    r_s = sample - hsc[t_s]
    cols = torch.arange(D, device=dev)
    w_idx = (wo[t_s] + r_s * D)[:, None] + cols  # [S, D] positions in the flat weights
    w_old = w.weights[w_idx].cpu().numpy()
    m_old = w.momentum[sample].cpu().numpy()
    # every lookup of a sampled row, grouped by row in lookup order
    pos = torch.isin(keys, sample).nonzero().squeeze(1)
    k = keys[pos]
    order = torch.sort(k, stable=True).indices
    pos, k = pos[order], k[order]
    b = bag[pos] % B
    g_rows = w.grad_output[b[:, None], (t_of[pos] * D)[:, None] + cols].cpu().numpy()  # [n, D]
    counts = torch.searchsorted(k, sample, right=True) - torch.searchsorted(k, sample)
    starts = np.concatenate([[0], np.cumsum(counts.cpu().numpy())])

    step()

    w_new = w.weights[w_idx].cpu().numpy()
    m_new = w.momentum[sample].cpu().numpy()
    for s in range(sample.numel()):
        n = int(starts[s + 1] - starts[s])
        if n == 0:  # untouched: bit-identical
            assert np.array_equal(w_new[s].view(np.uint16), w_old[s].view(np.uint16))
            assert m_new[s] == m_old[s]
            continue
        wt = np.ascontiguousarray(w_old[s]).copy()
        mt = np.array([m_old[s]], np.float32)
        oracle.backward(1, n, np.array([0, 1], np.int64), np.array([0, D], np.int32),
                        np.array([0], np.int64), wt, np.zeros(n, np.int64),
                        np.arange(n + 1, dtype=np.int64), g_rows[starts[s]:starts[s + 1]],
                        optimizer=oracle.ROWWISE_ADAGRAD, lr=w.lr, eps=w.eps, momentum=mt)
        np.testing.assert_allclose(m_new[s], mt[0], rtol=1e-4, atol=1e-5)
        if wt.dtype == np.float32:
            np.testing.assert_allclose(w_new[s], wt, rtol=1e-4, atol=1e-5)
        else:  # one ulp, or the derived bound of the device's fp32 arithmetic where it cancels
            one = synth.Workload(
                name="row", T=1, B=n, rows=np.array([1], np.int64), dims=np.array([D], np.int32),
                hash_size_cumsum=np.array([0, 1], np.int64), D_offsets=np.array([0, D], np.int32),
                weights_offsets=np.array([0], np.int64), momentum_offsets=None,
                weight_dtype=w.weight_dtype, grad_dtype=w.grad_dtype, optimizer=synth.ROWWISE_ADAGRAD,
                pooling=synth.SUM, nobag=False, lr=w.lr, eps=w.eps, indices=np.zeros(n, np.int64),
                offsets=np.arange(n + 1, dtype=np.int64), grad_output=g_rows[starts[s]:starts[s + 1]],
                weights=np.ascontiguousarray(w_old[s]), momentum=np.array([m_old[s]], np.float32))
            check16(one, oracle.ROWWISE_ADAGRAD, np.ascontiguousarray(w_new[s]), wt, one.weights,
                    one.momentum)
    return int(sample.numel())
