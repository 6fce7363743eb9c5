"""GPU parity of the forward pooled lookup: the CUDA path through the C ABI
against the oracle's forward, element by element on the same seeded inputs.

Bars: fp32 output within rtol 1e-4 / atol 1e-5 (fp32 sums against the
oracle's double sums, each rounded once). fp16 / bf16 output: within one ulp of
the output type plus the fp32 accumulation bound L * 2^-23 * sum_i |s_i w_i|
(a sum of signed terms can cancel to far below its terms, where one fp16 /
bf16 ulp is smaller than the fp32 rounding of the terms). Empty bags exactly
zero; errors reported as status.
"""
import numpy as np
import pytest

from _helpers import ATOL, MAX_ULP, RTOL, ulp_diff16
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
    rng = np.random.default_rng(seed + 2000)
    T = len(rows)
    lengths = lengths_fn(rng, T, B)
    ids_fn = ids_fn or (lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64))
    return synth.make_bag_workload("fwd", seed, rows, dims, B, lengths, ids_fn, **kw)


def run_forward(w, out_dtype=synth.F32, plan_kw=None):
    dw = dev.to_device(w)
    plan = dev.make_plan(w, **(plan_kw or {}))
    try:
        out = dev.forward(plan, dw, out_dtype=out_dtype)
        status = E.emb_plan_status(plan)
    finally:
        E.emb_plan_destroy(plan)
    got = out.cpu()
    if out_dtype == synth.BF16:
        got = got.view(__import__("torch").int16).numpy().view(np.uint16)
    else:
        got = got.numpy()
    return got, status


def expected(w, out_dtype=synth.F32):
    return oracle.forward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                          w.weights, w.indices, w.offsets, per_sample_weights=w.per_sample_weights,
                          mean=(w.pooling == synth.MEAN), out_dtype=out_dtype)


def as_f64(x, out_dtype):
    if out_dtype == synth.BF16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def check(w, out_dtype=synth.F32):
    got, status = run_forward(w, out_dtype)
    assert status == E.EMB_OK
    exp = expected(w, out_dtype)
    assert got.shape == exp.shape
    if out_dtype == synth.F32:
        np.testing.assert_allclose(got, exp, rtol=RTOL, atol=ATOL)
    else:
        d = ulp_diff16(got.view(np.uint16), exp.view(np.uint16))
        g64, e64 = as_f64(got, out_dtype), as_f64(exp, out_dtype)
        # one ulp of the output type at the expected value, plus the fp32 sum's bound
        ulp = np.abs(e64) * (2.0 ** (-10 if out_dtype == synth.F16 else -7)) + 1e-30
        absw = np.abs(w.weights.astype(np.float32)) if w.weight_dtype != synth.BF16 else \
            np.abs((w.weights.astype(np.uint32) << 16).view(np.float32))
        psw = None if w.per_sample_weights is None else np.abs(w.per_sample_weights)
        mag = oracle.forward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                             absw.astype(np.float32), w.indices, w.offsets, per_sample_weights=psw,
                             mean=(w.pooling == synth.MEAN)).astype(np.float64)
        Lmax = max(int(np.diff(w.offsets).max(initial=1)), 1)
        bound = ulp + Lmax * 2.0 ** -23 * mag
        bad = (d > MAX_ULP) & (np.abs(g64 - e64) > bound)
        assert not bad.any(), f"{bad.sum()} elements outside the bound (max ulp diff {d.max()})"
    empty = np.repeat(np.diff(w.offsets).reshape(w.T, w.B) == 0, w.dims, axis=0).T  # [B, sum D]
    assert np.all(got.astype(np.float32)[empty] == 0)
    return got


def test_tiny():
    check(synth.tiny(0))


def test_dlrm():
    check(synth.dlrm(0))


@pytest.mark.parametrize("odt", [synth.F32, synth.F16, synth.BF16])
def test_mixed_weighted_mean(odt):
    check(synth.mixed(0, B=2048), out_dtype=odt)


@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.SUM, True),
                                              (synth.MEAN, False), (synth.MEAN, True)])
@pytest.mark.parametrize("wdt", [synth.F32, synth.F16, synth.BF16])
def test_variants(pooling, weighted, wdt):
    w = custom(1, [300, 50, 2000], [8, 64, 20], 96, lambda r, T, B: r.integers(0, 40, (T, B)),
               pooling=pooling, weighted=weighted, weight_dtype=wdt)
    check(w)


@pytest.mark.parametrize("D", [4, 12, 128, 260, 1024, 4096])
def test_row_widths(D):
    # rows wider than one team's chunk are split into chunks
    w = custom(2, [64, 33], [D, D], 40, lambda r, T, B: r.integers(0, 30, (T, B)))
    check(w)


def test_empty_bags_and_long_bags():
    w = custom(3, [5000, 7], [32, 16], 300,
               lambda r, T, B: r.integers(0, 3, (T, B)) * (r.random((T, B)) < 0.3) + 600 * (r.random((T, B)) < 0.01))
    assert (np.diff(w.offsets) == 0).any() and np.diff(w.offsets).max() >= 600
    check(w)


def test_zero_lookups_writes_zeros():
    w = custom(4, [100, 100], [16, 16], 8, lambda r, T, B: np.zeros((T, B), np.int64))
    assert w.N == 0
    got = check(w)
    assert np.all(got == 0)


def test_forward_then_backward_adjoint_on_device():
    # <forward(W), g> over the batch equals <W_old - W_new, .> / lr under SGD: the
    # forward and the backward read the same lookups with the same scales
    w = custom(5, [400, 90], [32, 8], 64, lambda r, T, B: r.integers(0, 12, (T, B)),
               pooling=synth.MEAN, weighted=True, optimizer=synth.SGD, lr=1.0)
    dw = dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        out = dev.forward(plan, dw).cpu().numpy().astype(np.float64)
        w_old = dev.weights_numpy(dw).astype(np.float64)
        dev.step(plan, dw)
        assert E.emb_plan_status(plan) == E.EMB_OK
        w_new = dev.weights_numpy(dw).astype(np.float64)
    finally:
        E.emb_plan_destroy(plan)
    lhs = float(np.sum(out * w.grad_output.astype(np.float64)))
    rhs = float(np.dot(w_old, w_old - w_new))  # sum over rows of <W_row, G_row> (lr = 1)
    assert abs(lhs - rhs) <= 1e-3 * (abs(rhs) + 1.0)


def test_index_out_of_range_reported():
    w = custom(6, [100, 50], [16, 16], 20, lambda r, T, B: r.integers(1, 5, (T, B)))
    w.indices[-1] = 50  # one past the end of table 1
    got, status = run_forward(w)
    assert status == E.EMB_ERR_INDEX_OUT_OF_RANGE


def test_malformed_offsets_reported():
    w = custom(7, [100], [16], 20, lambda r, T, B: r.integers(1, 5, (T, B)))
    w.offsets[5], w.offsets[6] = w.offsets[6], w.offsets[5]  # one pair out of order
    got, status = run_forward(w)
    assert status == E.EMB_ERR_INVALID_ARG


def test_argument_errors():
    w = synth.tiny(0)
    dw = dev.to_device(w)
    plan = dev.make_plan(w)
    try:
        with pytest.raises(E.EmbError):  # batch above the plan's max_B
            E.emb_bag_fwd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B + 1, None, 0,
                          dw.weights, 0)
        with pytest.raises(E.EmbError):  # bad pooling mode
            E.emb_bag_fwd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B, None, 7,
                          dw.weights, 0)
    finally:
        E.emb_plan_destroy(plan)
