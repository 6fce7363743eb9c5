"""Pins for the oracle's forward pooled lookup against things other than itself.

* brute force: the output of table t as the dense product A_t W_t, where
  A_t[b, r] holds the summed scales of bag b's lookups of row r (numpy matmul);
* the adjoint identity with the backward: for any g, the sum over bags of
  <forward(W)_b, g_b> equals the sum over rows of <W_row, G_row>, with G the
  oracle's de-duplicated row gradients of g (a wrong scale, table offset or
  transposed index on either side breaks it);
* closed forms: an empty bag gives zeros, mean pooling of L copies of one row
  gives that row, a single weighted lookup gives psw times the row;
* storage rounding of the output (fp16 / bf16 bits of the double result) and
  the error codes.
"""
import numpy as np
import pytest

from sparse_embedding_bag_gb300 import synth


def small_workload(seed, nobag=False, maxlen=6, wdt=synth.F32):
    rng = np.random.default_rng(seed + 77)
    rows, dims, B = [7, 3, 11], [4, 8, 12], 5
    lengths = rng.integers(0, maxlen, (len(rows), B))
    return synth.make_bag_workload("pin", seed, rows, dims, B, lengths,
                                   lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                   weight_dtype=wdt, weighted=True)


def weights_f64(w):
    if w.weight_dtype == synth.BF16:
        return (w.weights.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return w.weights.astype(np.float64)


def brute_forward(w, psw=None, mean=False):
    W = weights_f64(w)
    out = np.zeros((w.B, int(w.D_offsets[-1])))
    for t in range(w.T):
        E, D = int(w.rows[t]), int(w.dims[t])
        A = np.zeros((w.B, E))
        for b in range(w.B):
            bt = t * w.B + b
            L = int(w.offsets[bt + 1] - w.offsets[bt])
            for i in range(int(w.offsets[bt]), int(w.offsets[bt + 1])):
                s = 1.0 if psw is None else float(psw[i])
                if mean:
                    s /= L
                A[b, int(w.indices[i])] += s
        Wt = W[int(w.weights_offsets[t]):int(w.weights_offsets[t]) + E * D].reshape(E, D)
        out[:, int(w.D_offsets[t]):int(w.D_offsets[t + 1])] = A @ Wt
    return out


def fwd(oracle_mod, w, psw=None, mean=False, out_dtype=None):
    return oracle_mod.forward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                              w.weights, w.indices, w.offsets, per_sample_weights=psw, mean=mean,
                              out_dtype=oracle_mod.F32 if out_dtype is None else out_dtype)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", ["sum", "mean", "weighted", "weighted_mean"])
def test_forward_vs_one_hot_matmul(oracle_mod, seed, mode):
    w = small_workload(seed)
    psw = w.per_sample_weights if "weighted" in mode else None
    got = fwd(oracle_mod, w, psw=psw, mean="mean" in mode)
    exp = brute_forward(w, psw=psw, mean="mean" in mode)
    np.testing.assert_allclose(got.astype(np.float64), exp.astype(np.float32).astype(np.float64),
                               rtol=2e-7, atol=1e-9)


def test_forward_tiny_config_vs_one_hot(oracle_mod):
    w = synth.tiny(0)
    np.testing.assert_allclose(fwd(oracle_mod, w).astype(np.float64), brute_forward(w),
                               rtol=2e-7, atol=1e-9)


@pytest.mark.parametrize("mode", ["sum", "mean", "weighted_mean"])
def test_forward_is_adjoint_of_backward(oracle_mod, mode):
    w = small_workload(9, maxlen=8)
    psw = w.per_sample_weights if "weighted" in mode else None
    mean = "mean" in mode
    out = fwd(oracle_mod, w, psw=psw, mean=mean).astype(np.float64)
    g = w.grad_output.astype(np.float64)
    lhs = float(np.sum(out * g))
    keys, G = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices,
                                   w.offsets, w.grad_output, per_sample_weights=psw, mean=mean)
    W = weights_f64(w)
    rhs = 0.0
    for r, k in enumerate(keys):
        t = int(np.searchsorted(w.hash_size_cumsum, k, side="right") - 1)
        D = int(w.dims[t])
        row = W[int(w.weights_offsets[t]) + (k - int(w.hash_size_cumsum[t])) * D:][:D]
        rhs += float(np.dot(row, G[r, :D]))
    assert abs(lhs - rhs) <= 1e-5 * (abs(rhs) + 1.0)


def test_forward_closed_forms(oracle_mod):
    rows, dims, B = [6], [8], 4
    lengths = np.array([[0, 3, 1, 5]])
    ids = [np.array([2, 2, 2, 4, 1, 1, 1, 1, 1], np.int64)]
    w = synth.make_bag_workload("closed", 0, rows, dims, B, lengths, lambda r, t, n: ids[t][:n])
    W = w.weights.reshape(6, 8).astype(np.float64)
    out = fwd(oracle_mod, w, mean=True)
    assert np.all(out[0] == 0.0)                             # empty bag
    np.testing.assert_array_equal(out[1], W[2].astype(np.float32))  # mean of three copies
    np.testing.assert_array_equal(out[2], W[4].astype(np.float32))
    np.testing.assert_array_equal(out[3], W[1].astype(np.float32))
    psw = np.full(w.N, 0.5, np.float32)
    out_w = fwd(oracle_mod, w, psw=psw)
    np.testing.assert_array_equal(out_w[2], (0.5 * W[4]).astype(np.float32))  # one weighted lookup


@pytest.mark.parametrize("odt", ["f16", "bf16"])
def test_forward_output_rounding(oracle_mod, odt):
    w = small_workload(4)
    exp = brute_forward(w)
    code = oracle_mod.F16 if odt == "f16" else oracle_mod.BF16
    got = fwd(oracle_mod, w, out_dtype=code)
    conv = oracle_mod.double_to_half_bits if odt == "f16" else oracle_mod.double_to_bf16_bits
    bits = got.view(np.uint16) if odt == "f16" else got
    # the oracle rounds its double sum once; the brute-force sum may differ in the last
    # double bits, so compare the rounded values allowing a one-step difference
    for e, b in zip(exp.ravel(), bits.ravel()):
        assert abs(int(conv(e)) - int(b)) <= 1


def test_forward_bf16_weights_vs_one_hot(oracle_mod):
    w = small_workload(5, wdt=synth.BF16)
    np.testing.assert_allclose(fwd(oracle_mod, w).astype(np.float64), brute_forward(w),
                               rtol=2e-7, atol=1e-9)


def test_forward_error_codes(oracle_mod):
    w = small_workload(6)
    bad = w.indices.copy()
    assert w.offsets[w.B] > 0  # table 0 has lookups, so lookup 0 is one of them
    bad[0] = w.rows[0]  # one past the end of table 0
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.forward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                           w.weights, bad, w.offsets)
    assert e.value.code == 3
    off = w.offsets.copy()
    off[-1] += 1
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.forward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                           w.weights, w.indices, off)
    assert e.value.code == 1
