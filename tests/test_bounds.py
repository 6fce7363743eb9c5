"""The derived error bound of tests/_bounds.py against fp32 evaluations of the
same updates done here in numpy (several summation orders: in lookup order,
reversed, shuffled, pairwise, and the row-wise sum of squares by chunks as rows
wider than one chunk take it), including updates that cancel; and its size where
nothing cancels (well below one 16-bit spacing of the operands, so the 16-bit bars
stay at one ulp there)."""
import numpy as np
import pytest

from _bounds import ADAGRAD, ROWWISE_ADAGRAD, SGD, _lookups, spacing16, to_f64, update_bounds
from sparse_embedding_bag_gb300 import synth

f32 = np.float32


def fma32(a, b, c):
    # a*b is exact in double for fp32 operands; the sum is rounded once to double,
    # then to fp32 (a double rounding that differs from one rounding only in
    # ties of measure zero here)
    return f32(np.float64(a) * np.float64(b) + np.float64(c))


def fp32_sum(terms, order):
    if order == "pairwise":
        vals = [f32(x) for x in terms]
        while len(vals) > 1:
            vals = [f32(vals[i] + vals[i + 1]) if i + 1 < len(vals) else vals[i] for i in range(0, len(vals), 2)]
        return vals[0]
    acc = f32(0)
    for x in terms:
        acc = f32(acc + x)
    return acc


def device_like_update(w, opt, K, order, rng, w_old, m_old):
    """The fp32 update of row K the way the device evaluates it (any summation order)."""
    keys, _, grow, _ = _lookups(w)
    pos = np.nonzero(keys == K)[0]
    hsc = w.hash_size_cumsum
    t = int(np.searchsorted(hsc, K, side="right") - 1)
    D = int(w.dims[t])
    Do = w.D_offsets
    off = np.asarray(w.offsets)
    L = np.diff(off)[np.repeat(np.arange(w.T * w.B), np.diff(off))]
    G = np.zeros(D, f32)
    for d in range(D):
        terms = []
        for i in pos:
            g = f32(to_f64(np.asarray(w.grad_output)[grow[i], Do[t] + d:Do[t] + d + 1], w.grad_dtype)[0])
            s = f32(1.0)
            if w.per_sample_weights is not None:
                s = f32(w.per_sample_weights[i])
            if w.pooling == synth.MEAN:
                s = f32(s / f32(L[i]))
            terms.append(fma32(s, g, 0.0))
        if order == "reversed":
            terms = terms[::-1]
        elif order == "shuffled":
            terms = [terms[j] for j in rng.permutation(len(terms))]
        G[d] = fp32_sum(terms, order)
    o = int(w.weights_offsets[t]) + int(K - hsc[t]) * D
    wrow = to_f64(np.asarray(w_old)[o:o + D], w.weight_dtype).astype(f32)
    lr, eps = f32(w.lr), f32(w.eps)
    if opt == SGD:
        return np.array([fma32(-lr, G[d], wrow[d]) for d in range(D)])
    if opt == ROWWISE_ADAGRAD:
        sq = [fma32(G[d], G[d], 0.0) for d in range(D)]
        if order == "chunked":  # a row of several chunks: each chunk's sum, then the sums in chunk order
            ss = fp32_sum([fp32_sum(sq[c:c + 4], "forward") for c in range(0, D, 4)], "forward")
        else:
            ss = fp32_sum(sq, order)
        m = f32(f32(m_old[K]) + f32(ss / f32(D)))
        mult = f32(lr / f32(f32(np.sqrt(m)) + eps))
        return np.array([fma32(-mult, G[d], wrow[d]) for d in range(D)])
    out = []
    for d in range(D):
        m = fma32(G[d], G[d], f32(m_old[o + d]))
        mult = f32(lr / f32(f32(np.sqrt(m)) + eps))
        out.append(fma32(-mult, G[d], wrow[d]))
    return np.array(out)


def small(seed, opt, wdt, cancel=False):
    rng = np.random.default_rng(seed)
    rows, dims, B = [40, 25], [8, 12], 24
    w = synth.make_bag_workload("bounds", seed, rows, dims, B, rng.integers(1, 12, (2, B)),
                                lambda r, t, n: r.integers(0, 6, n).astype(np.int64),
                                weight_dtype=wdt, optimizer=opt if opt != ADAGRAD else synth.SGD,
                                pooling=synth.MEAN, weighted=True, lr=0.05, eps=1e-4)
    if cancel:
        # the old weights equal the step (computed in double), so w - step cancels
        keys, _, grow, s = _lookups(w)
        g = to_f64(np.asarray(w.grad_output), w.grad_dtype)
        for K in np.unique(keys):
            t = int(np.searchsorted(w.hash_size_cumsum, K, side="right") - 1)
            D = int(w.dims[t])
            pos = keys == K
            G = (s[pos][:, None] * g[grow[pos]][:, w.D_offsets[t]:w.D_offsets[t + 1]]).sum(0)
            o = int(w.weights_offsets[t]) + int(K - w.hash_size_cumsum[t]) * D
            w.weights[o:o + D] = (w.lr * G).astype(np.float16 if wdt == synth.F16 else np.float32)
    return w


@pytest.mark.parametrize("opt", [SGD, ROWWISE_ADAGRAD, ADAGRAD])
@pytest.mark.parametrize("cancel", [False, True])
def test_bound_covers_fp32_evaluations(opt, cancel):
    rng = np.random.default_rng(1)
    w = small(3, opt, synth.F16 if opt != ADAGRAD or not cancel else synth.F32, cancel)
    m_rows = np.full(int(w.hash_size_cumsum[-1]), 0.3, np.float32)
    m_elems = np.full(np.asarray(w.weights).size, 0.3, np.float32)
    m_old = m_rows if opt == ROWWISE_ADAGRAD else m_elems if opt == ADAGRAD else None
    keys = np.unique(_lookups(w)[0])
    bounds = update_bounds(w, opt, keys, w.weights, m_old)
    worst = 0.0
    for K, (eps, x) in zip(keys, bounds):
        for order in ("forward", "reversed", "shuffled", "pairwise", "chunked"):
            got = device_like_update(w, opt, K, order, rng, w.weights, m_old).astype(np.float64)
            err = np.abs(got - x)
            assert np.all(err <= eps), (K, order, (err / eps).max())
            worst = max(worst, float((err / eps).max()))
    assert worst > 1e-3  # the bound is not vacuous: the evaluations come within its scale


def test_bound_is_far_below_one_spacing_of_the_operands():
    # the bound scales with the operands w and step, not with their difference:
    # against the spacing at |w| + |step| it stays well below one spacing, so where
    # w - step does not cancel, a bar of one spacing plus the bound still admits
    # exactly one ulp (16-bit differences are whole spacings)
    w = small(4, ROWWISE_ADAGRAD, synth.F16)
    m_old = np.full(int(w.hash_size_cumsum[-1]), 0.3, np.float32)
    keys = np.unique(_lookups(w)[0])
    for K, (eps, x) in zip(keys, update_bounds(w, ROWWISE_ADAGRAD, keys, w.weights, m_old)):
        t = int(np.searchsorted(w.hash_size_cumsum, K, side="right") - 1)
        D = int(w.dims[t])
        o = int(w.weights_offsets[t]) + int(K - w.hash_size_cumsum[t]) * D
        wrow = to_f64(w.weights[o:o + D], w.weight_dtype)
        mag = np.abs(wrow) + np.abs(wrow - x)
        assert np.all(eps < 0.25 * spacing16(mag, synth.F16))
