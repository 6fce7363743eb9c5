"""Pins for the oracle's elementwise Adagrad and dense-gradient mode against
things other than themselves.

* elementwise Adagrad on hand-worked dyadic values (eps = 0): from a zero state
  one step moves every element by lr * sign(g);
* with D = 1 the elementwise and the row-wise Adagrad coincide (the row mean of
  g^2 over one element is g^2): two different oracle routines must agree bitwise;
* dense gradients equal the brute-force one-hot products A_t^T g_t on touched
  rows and are exactly zero elsewhere (sum, mean, weighted, unpooled).
"""
import numpy as np
import pytest

from sparse_embedding_bag_gb300 import synth
from test_oracle_pins import brute_force_G, small_workload


def test_adagrad_hand_values(oracle_mod):
    w = np.ones(4, np.float32)
    m = np.zeros(4, np.float32)
    g = np.array([2.0, -8.0, 0.5, 16.0])
    oracle_mod.apply_row(oracle_mod.ADAGRAD, w, 0, 4, g, momentum=m, momentum_index=0,
                         lr=0.25, eps=0.0)
    # m = g^2; w = 1 - 0.25 * g / |g|
    assert m.tolist() == [4.0, 64.0, 0.25, 256.0]
    assert w.tolist() == [0.75, 1.25, 0.75, 0.75]
    # from state 9 with g = 4: m = 25, w = 3 - 0.5 * 4 / 5 = 2.6, rounded once to fp32
    w2 = np.array([3.0], np.float32)
    m2 = np.array([9.0], np.float32)
    oracle_mod.apply_row(oracle_mod.ADAGRAD, w2, 0, 1, np.array([4.0]), momentum=m2, lr=0.5, eps=0.0)
    assert m2.tolist() == [25.0] and w2[0] == np.float32(2.6)


def test_adagrad_equals_rowwise_for_one_element_rows(oracle_mod):
    # with D = 1 the row mean of g^2 is g^2, and the weights layout equals the
    # row-wise state layout (weights_offsets == hash_size_cumsum)
    rows, B = [40, 25], 32
    lengths = np.random.default_rng(2).integers(0, 5, (2, B))
    w1 = synth.make_bag_workload("d1", 4, rows, [1, 1], B, lengths,
                                 lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64))
    assert np.array_equal(w1.weights_offsets, w1.hash_size_cumsum[:-1])
    outs = []
    for opt in (oracle_mod.ROWWISE_ADAGRAD, oracle_mod.ADAGRAD):
        weights = w1.weights.copy()
        mom = np.full(int(w1.hash_size_cumsum[-1]), 0.5, np.float32)
        oracle_mod.backward(w1.T, w1.B, w1.hash_size_cumsum, w1.D_offsets, w1.weights_offsets,
                            weights, w1.indices, w1.offsets, w1.grad_output, optimizer=opt,
                            lr=0.05, eps=1e-3, momentum=mom)
        outs.append((weights, mom))
    assert not np.array_equal(outs[0][0], w1.weights)  # something was updated
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))


@pytest.mark.parametrize("mode", ["sum", "mean", "weighted", "nobag"])
def test_dense_grad_vs_one_hot(oracle_mod, mode):
    nobag = mode == "nobag"
    w = small_workload(21, nobag=nobag)
    psw = w.per_sample_weights if mode == "weighted" else None
    extent = int(w.weights.size)
    out = oracle_mod.dense_grad(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                                extent, w.indices, w.offsets, w.grad_output,
                                per_sample_weights=psw, mean=(mode == "mean"), nobag=nobag)
    Gs = brute_force_G(w, psw=psw, mean=(mode == "mean"), nobag=nobag)
    for t in range(w.T):
        E, D = int(w.rows[t]), int(w.dims[t])
        o = int(w.weights_offsets[t])
        got = out[o:o + E * D].reshape(E, D).astype(np.float64)
        touched, G = Gs[t]
        np.testing.assert_allclose(got[touched], G[touched].astype(np.float32), rtol=2e-7, atol=1e-9)
        assert np.all(got[~touched] == 0.0)
