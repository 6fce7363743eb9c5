"""GPU parity of elementwise Adagrad and of the dense-gradient mode: the CUDA
path through the C ABI against the oracle on the same seeded inputs.

Bars: fp32 weights, state and gradients within rtol 1e-4 / atol 1e-5;
fp16 / bf16 weights within 1 ulp of the oracle's rounded value (an update
w - lr * g / (sqrt(m) + eps) moves w by less than lr, so it does not cancel);
fp16 / bf16 dense gradients within one ulp plus the fp32 accumulation bound
L * 2^-23 * sum |s g| of the row (a row's gradient is a signed sum that can
cancel); untouched rows bit-identical (updates) or exactly zero (dense).
"""
import numpy as np
import pytest

from _bounds import check16
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
    rng = np.random.default_rng(seed + 3000)
    T = len(rows)
    lengths = lengths_fn(rng, T, B)
    ids_fn = ids_fn or (lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64))
    return synth.make_bag_workload("da", seed, rows, dims, B, lengths, ids_fn, **kw)


def to_f64(x, dtype):
    if dtype == synth.BF16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# ---------------------------------------------------------------- elementwise Adagrad

def run_adagrad(w, m0):
    import torch
    dw = dev.to_device(w)
    mom = torch.from_numpy(m0.copy()).cuda()
    plan = dev.make_plan(w)
    try:
        E.emb_bag_bwd_adagrad(plan, dw.weights, mom, dw.indices, dw.offsets, w.N, w.B,
                              dw.per_sample_weights, dw.grad_output, w.pooling, w.lr, w.eps)
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)
    return dev.weights_numpy(dw), mom.cpu().numpy()


def check_adagrad(w, m_init=0.25):
    m0 = np.full(w.weights.size, m_init, np.float32)
    got_w, got_m = run_adagrad(w, m0)
    exp_w, exp_m = np.array(w.weights, copy=True), m0.copy()
    oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, exp_w,
                    w.indices, w.offsets, w.grad_output, optimizer=oracle.ADAGRAD, lr=w.lr,
                    eps=w.eps, momentum=exp_m, per_sample_weights=w.per_sample_weights,
                    mean=(w.pooling == synth.MEAN), grad_dtype=w.grad_dtype)
    np.testing.assert_allclose(got_m, exp_m, rtol=RTOL, atol=ATOL)
    untouched = exp_m == m0
    assert np.array_equal(got_m[untouched], m0[untouched])
    if got_w.dtype == np.float32:
        np.testing.assert_allclose(got_w, exp_w, rtol=RTOL, atol=ATOL)
    else:  # one ulp, or the derived bound where an update cancels
        check16(w, oracle.ADAGRAD, got_w, exp_w, w.weights, m0)


def test_adagrad_dlrm():
    w = synth.dlrm(3)
    check_adagrad(w)


@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.MEAN, True)])
@pytest.mark.parametrize("wdt", [synth.F32, synth.F16, synth.BF16])
def test_adagrad_variants(pooling, weighted, wdt):
    w = custom(1, [300, 50, 2000], [8, 64, 20], 96, lambda r, T, B: r.integers(0, 40, (T, B)),
               pooling=pooling, weighted=weighted, weight_dtype=wdt)
    check_adagrad(w)


@pytest.mark.parametrize("D", [4, 132, 1028, 4096])
def test_adagrad_row_widths(D):
    # elementwise state: rows of any width, also those split into chunks
    w = custom(2, [40, 17], [D, D], 30, lambda r, T, B: r.integers(0, 40, (T, B)))
    check_adagrad(w)


def test_adagrad_hot_rows_split_over_warps():
    w = custom(3, [1000], [64], 4096, lambda r, T, B: r.integers(20, 60, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.5, 0, r.integers(0, 1000, n)).astype(np.int64))
    check_adagrad(w)


# ---------------------------------------------------------------- dense gradient

def run_dense(w, out_dtype_np):
    import torch
    dw = dev.to_device(w)
    tdt = {np.float32: torch.float32, np.float16: torch.float16, np.uint16: torch.bfloat16}[out_dtype_np]
    buf = torch.full((w.weights.size,), 7.0, dtype=tdt, device="cuda")  # non-zero: must be cleared
    plan = dev.make_plan(w, max_N=max(w.N, 16))
    try:
        if w.nobag:
            E.emb_nobag_bwd_dense_grad(plan, buf, dw.indices, dw.offsets, w.N, w.B, dw.grad_output)
        else:
            E.emb_bag_bwd_dense_grad(plan, buf, dw.indices, dw.offsets, w.N, w.B,
                                     dw.per_sample_weights, dw.grad_output, w.pooling)
        assert E.emb_plan_status(plan) == E.EMB_OK
    finally:
        E.emb_plan_destroy(plan)
    got = buf.cpu()
    if out_dtype_np == np.uint16:
        return got.view(torch.int16).numpy().view(np.uint16)
    return got.numpy()


def check_dense(w):
    odt = {synth.F32: oracle.F32, synth.F16: oracle.F16, synth.BF16: oracle.BF16}[w.weight_dtype]
    np_dt = {synth.F32: np.float32, synth.F16: np.float16, synth.BF16: np.uint16}[w.weight_dtype]
    got = run_dense(w, np_dt)
    kw = dict(per_sample_weights=w.per_sample_weights, mean=(w.pooling == synth.MEAN),
              nobag=w.nobag, grad_dtype=w.grad_dtype)
    exp = oracle.dense_grad(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                            w.weights.size, w.indices, w.offsets, w.grad_output, out_dtype=odt, **kw)
    if np_dt == np.float32:
        np.testing.assert_allclose(got, exp, rtol=RTOL, atol=ATOL)
    else:
        g64, e64 = to_f64(got, w.weight_dtype), to_f64(exp, w.weight_dtype)
        d = ulp_diff16(got.view(np.uint16), exp.view(np.uint16))
        ulp = np.abs(e64) * (2.0 ** (-10 if w.weight_dtype == synth.F16 else -7)) + 1e-30
        gabs = np.abs(to_f64(np.asarray(w.grad_output), w.grad_dtype)).astype(np.float32)
        kw2 = dict(kw, grad_dtype=None,
                   per_sample_weights=None if w.per_sample_weights is None else np.abs(w.per_sample_weights))
        mag = oracle.dense_grad(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                                w.weights.size, w.indices, w.offsets, gabs, **kw2).astype(np.float64)
        bad = (d > MAX_ULP) & (np.abs(g64 - e64) > ulp + w.N * 2.0 ** -23 * mag)
        assert not bad.any(), f"{bad.sum()} elements outside the bound (max ulp diff {d.max()})"
    # rows no lookup touched are exactly zero (the oracle's zeros are exact too)
    touched_keys = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, 32)["run_keys"]
    mask = np.zeros(w.weights.size, bool)
    for k in touched_keys:
        t = int(np.searchsorted(w.hash_size_cumsum, k, side="right") - 1)
        D = int(w.dims[t])
        o = int(w.weights_offsets[t]) + (int(k) - int(w.hash_size_cumsum[t])) * D
        mask[o:o + D] = True
    assert np.all(to_f64(got, w.weight_dtype)[~mask] == 0)


def test_dense_dlrm():
    check_dense(synth.dlrm(4))


@pytest.mark.parametrize("pooling,weighted", [(synth.SUM, False), (synth.SUM, True),
                                              (synth.MEAN, False), (synth.MEAN, True)])
@pytest.mark.parametrize("wdt", [synth.F32, synth.F16, synth.BF16])
def test_dense_variants(pooling, weighted, wdt):
    w = custom(5, [300, 50, 2000], [8, 64, 20], 96, lambda r, T, B: r.integers(0, 40, (T, B)),
               pooling=pooling, weighted=weighted, weight_dtype=wdt)
    check_dense(w)


@pytest.mark.parametrize("D", [64, 4096])
def test_dense_unpooled(D):
    w = custom(6, [100, 3000, 17], [D, D, D], 3, lambda r, T, B: r.integers(0, 60, (T, B)),
               nobag=True)
    check_dense(w)


def test_dense_zero_lookups_clears_buffer():
    w = custom(7, [100, 100], [16, 16], 8, lambda r, T, B: np.zeros((T, B), np.int64))
    assert w.N == 0
    got = run_dense(w, np.float32)
    assert np.all(got == 0)
