"""A-priori bounds on the device's fp32 rounding error in a weight update, for
the parity bars of 16-bit weights.

The device computes a row's gradient G as an fp32 sum of the run's n terms
s_i * g_i (each term an fma of the fp32 scale s_i = fl(psw_i / L) with the
gradient value, which converts to fp32 exactly), in some order of its own: lane
groups add their lookups in turn, groups are folded by shuffles, pieces of a run
cut by slice ends are added as fp32 partial rows. Whatever that order, it is a
binary tree of at most n roundings on every path from a term to the root, plus
one rounding of each scale, so (Higham, "Accuracy and Stability of Numerical
Algorithms", 2nd ed., section 4.2, with gamma_k = k u / (1 - k u), u = 2^-24)

    |G_dev - G| <= gamma_{n+1} * sum_i |s_i g_i|            (elementwise)

The update then rounds a few more times in fp32: the row-wise Adagrad state
m + sum(G^2)/D (a D-term sum of squares, a division and an addition), its
square root, the addition of eps, the division lr / (...), and the final
fma w - mult * G; elementwise Adagrad rounds m + G^2 (one fma) and the same
chain per element. Each step's error is carried through in double below, so
the result bounds |x_dev - x| for the fp32 update x_dev against the exact
update x = w - mult * G.

The 16-bit bars follow from it:
* round to nearest: RN moves each side by at most half a spacing, so
  |got - exp| <= sp + eps with sp the spacing of the format at |x| + eps;
* stochastic rounding: the device rounds x_dev to one end of its bracket and
  the oracle rounds fl32(x) to one end of its own, so
  |got - exp| <= 2 sp + eps + u |x| (spacing at |x| + eps + u |x|).
Where w - step does not cancel, eps is far below one spacing and the bars
reduce to one (RN) or two (SR) ulps; where it cancels, the fp32 error of the
step, which does not shrink with the result, is what eps accounts for.
"""
import numpy as np

from sparse_embedding_bag_gb300 import synth

U = 2.0 ** -24  # fp32 unit roundoff
SGD, ROWWISE_ADAGRAD, ADAGRAD = 0, 1, 2


def gamma(k):
    k = np.asarray(k, np.float64)
    return k * U / (1.0 - k * U)


def to_f64(x: np.ndarray, dtype: int) -> np.ndarray:
    """Storage values (bf16 as uint16 bits) as doubles."""
    if dtype == synth.BF16:
        return (np.asarray(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x).astype(np.float64)


def spacing16(v: np.ndarray, dtype: int) -> np.ndarray:
    """Distance between consecutive fp16 / bf16 values at magnitude |v| (the binade's ulp)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 1e-300)
    e = np.floor(np.log2(a))
    if dtype == synth.F16:
        return 2.0 ** (np.maximum(e, -14.0) - 10.0)
    return 2.0 ** (np.maximum(e, -126.0) - 7.0)


def _lookups(w):
    """Per lookup: linear index, table, gradient row, exact scale (double)."""
    off = np.asarray(w.offsets, np.int64)
    lengths = np.diff(off)
    bt = np.repeat(np.arange(w.T * w.B), lengths)
    t = bt // w.B
    keys = np.asarray(w.hash_size_cumsum, np.int64)[t] + np.asarray(w.indices, np.int64)
    grow = np.arange(keys.size) if w.nobag else bt % w.B
    s = np.ones(keys.size)
    if w.per_sample_weights is not None:
        s = np.asarray(w.per_sample_weights, np.float64).copy()
    if w.pooling == synth.MEAN and not w.nobag:
        s = s / lengths[bt]
    return keys, t, grow, s


def _mult(lr, eps, m, e_m):
    """lr / (sqrt(m) + eps) and a bound on the error of its fp32 evaluation from m +- e_m."""
    r = np.sqrt(m)
    with np.errstate(divide="ignore", invalid="ignore"):
        e_r = np.minimum(np.sqrt(e_m), np.where(r > 0, e_m / np.where(r > 0, r, 1.0), np.inf))
    e_r = e_r + U * (r + e_r)                      # the square root's own rounding
    den = r + eps
    e_den = e_r + U * (den + e_r)                  # the addition of eps
    assert np.all(den > e_den), "denominator bound not positive"
    mult = lr / den
    e_mult = lr * e_den / (den * (den - e_den)) + U * lr / (den - e_den)  # and the division
    return mult, e_mult


def update_bounds(w, opt, keys_sel, w_old, m_old=None):
    """For every linear index in keys_sel: (eps[D], x[D]) with x the exact update
    w - step (double) and eps a bound on |device fp32 update - x|.
    w_old: the flat weights before the step (storage representation); m_old: the
    state before the step (row-wise: one per linear index / momentum offset;
    elementwise: laid out like the weights)."""
    keys, tl, grow, s = _lookups(w)
    hsc = np.asarray(w.hash_size_cumsum, np.int64)
    Do = np.asarray(w.D_offsets, np.int64)
    g_all = w.grad_output
    lr, eps_ = float(np.float32(w.lr)), float(np.float32(w.eps))
    out = []
    for K in np.asarray(keys_sel, np.int64):
        pos = np.nonzero(keys == K)[0]
        t = int(np.searchsorted(hsc, K, side="right") - 1)
        idx = int(K - hsc[t])
        D = int(Do[t + 1] - Do[t])
        n = pos.size
        if w.nobag:
            gs = to_f64(np.asarray(g_all)[grow[pos]], w.grad_dtype)
        else:
            gs = to_f64(np.asarray(g_all)[grow[pos]][:, Do[t]:Do[t + 1]], w.grad_dtype)
        sv = s[pos][:, None]
        G = (sv * gs).sum(0)
        eG = gamma(n + 1) * (np.abs(sv) * np.abs(gs)).sum(0)
        o = int(w.weights_offsets[t]) + idx * D
        wrow = to_f64(np.asarray(w_old)[o:o + D], w.weight_dtype)
        if opt == SGD:
            mult, e_mult = lr, 0.0
        elif opt == ROWWISE_ADAGRAD:
            mo = w.momentum_offsets
            m0 = float(m_old[(int(mo[t]) if mo is not None else int(hsc[t])) + idx])
            ss = float((G * G).sum())
            e_ss = float((2 * np.abs(G) * eG + eG * eG).sum() + gamma(D) * ((np.abs(G) + eG) ** 2).sum())
            m = m0 + ss / D
            e_m = e_ss / D + gamma(2) * (m0 + (ss + e_ss) / D)
            mult, e_mult = _mult(lr, eps_, m, e_m)
        else:
            m0 = np.asarray(m_old[o:o + D], np.float64)
            m = m0 + G * G
            e_m = 2 * np.abs(G) * eG + eG * eG
            e_m = e_m + U * (m + e_m)
            mult, e_mult = _mult(lr, eps_, m, e_m)
        x = wrow - mult * G
        e_step = mult * eG + np.abs(G) * e_mult + e_mult * eG
        out.append((e_step + U * (np.abs(x) + e_step), x))  # the final fma's rounding
    return out


def check16(w, opt, got, exp, w_old, m_old=None, sr=False):
    """16-bit weight updates (got, exp: flat storage arrays; w_old, m_old: the
    weights and state before the step): every element that differs from the
    oracle's by more than one ulp must lie within the derived bar (one spacing
    plus eps for round to nearest; two spacings plus eps + u |x| for stochastic
    rounding). Elements at most one ulp apart pass without computing a bound.
    Returns the number of elements that needed the bound."""
    from _helpers import ulp_diff16
    gb, eb = np.asarray(got).view(np.uint16), np.asarray(exp).view(np.uint16)
    far = np.nonzero(ulp_diff16(gb, eb) > 1)[0]
    if far.size == 0:
        return 0
    rows = _element_rows(w, far)
    sel = np.unique(rows)
    bounds = dict(zip(sel.tolist(), update_bounds(w, opt, sel, w_old, m_old)))
    for e_i, K in zip(far, rows):
        _, o = _elem_pos(w, K)
        eps, x = bounds[int(K)]
        d = int(e_i - o)
        g64 = to_f64(np.asarray(got)[e_i:e_i + 1], w.weight_dtype)[0]
        e64 = to_f64(np.asarray(exp)[e_i:e_i + 1], w.weight_dtype)[0]
        if sr:
            err = eps[d] + U * abs(x[d])
            bar = 2 * spacing16(abs(x[d]) + err, w.weight_dtype) + err
        else:
            bar = spacing16(abs(x[d]) + eps[d], w.weight_dtype) + eps[d]
        assert abs(g64 - e64) <= bar, (f"row {int(K)} element {d}: |{g64} - {e64}| = {abs(g64 - e64)} "
                                       f"beyond the derived bound {bar}")
    return int(far.size)


def _element_rows(w, flat_idx):
    """Linear index of the row that holds each flat weights element."""
    hsc = np.asarray(w.hash_size_cumsum, np.int64)
    wo = np.asarray(w.weights_offsets, np.int64)
    dims = np.asarray(w.dims, np.int64)
    out = np.empty(flat_idx.size, np.int64)
    for k, e in enumerate(flat_idx):
        cand = np.nonzero((wo <= e) & (e < wo + (hsc[1:] - hsc[:-1]) * dims))[0]
        assert cand.size == 1
        t = int(cand[0])
        out[k] = hsc[t] + (e - wo[t]) // dims[t]
    return out


def _elem_pos(w, K):
    hsc = np.asarray(w.hash_size_cumsum, np.int64)
    t = int(np.searchsorted(hsc, K, side="right") - 1)
    D = int(w.dims[t])
    return t, int(w.weights_offsets[t]) + int(K - hsc[t]) * D
