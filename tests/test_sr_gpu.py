"""GPU parity of stochastic rounding of fp16 / bf16 weight stores: the CUDA path
through the C ABI against the oracle with the same seed and call number.

Both sides draw the same Philox4x32-10 words and take the same rounding rule,
so they agree bit for bit except where the fp32 update computed on the device
and the oracle's update (double, rounded once to fp32) differ by a few fp32
ulps and a random word falls between the two thresholds: a chance of about
2^-13 per fp16 element and 2^-16 per bf16 element. The bar: at most 0.5% of the
touched elements differ; an element that differs by more than one ulp must lie
within two spacings of the format plus the a-priori bound of the device's fp32
update (its summation of the run's terms and the optimizer's roundings, derived
in tests/_bounds.py): each side rounds to one end of its own bracket, and the
brackets can differ when the two fp32 updates lie on either side of a
representable value, or, where w - step cancels, by more than one spacing.
Untouched rows are bit-identical. Properties that hold at any size: the rounding is unbiased
(the share of roundings away from zero matches the dropped fraction), a
second run with the same seed and call is bit-identical, and the call number
advances by one per update call.
"""
import numpy as np
import pytest

from _bounds import check16
from _helpers import ulp_diff16
import oracle
from sparse_embedding_bag_gb300 import device as dev
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import synth

pytestmark = pytest.mark.gpu

SR = E.EMB_FLAG_STOCHASTIC_ROUNDING
MAX_MISMATCH = 0.005


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_embedding_bag_gb300 import build
    build.build()
    E.load()


def custom(seed, rows, dims, B, lengths_fn, ids_fn=None, **kw):
    rng = np.random.default_rng(seed + 4000)
    lengths = lengths_fn(rng, len(rows), B)
    ids_fn = ids_fn or (lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64))
    return synth.make_bag_workload("sr", seed, rows, dims, B, lengths, ids_fn, **kw)


def state_init(w, opt):
    if opt == oracle.ROWWISE_ADAGRAD:
        return np.full(int(w.hash_size_cumsum[-1]), 0.25, np.float32)
    if opt == oracle.ADAGRAD:
        return np.full(w.weights.size, 0.25, np.float32)
    return None


def gpu_update(w, opt, flags, seed=0, call=0, calls=1, weights=None, m0=None):
    """Runs `calls` update calls; returns (weights, state, plan's seed and next call)."""
    import torch
    if weights is not None:
        w.weights = weights
    dw = dev.to_device(w)
    mom = None if m0 is None else torch.from_numpy(m0.copy()).cuda()
    plan = dev.make_plan(w, flags=flags)
    try:
        E.emb_plan_set_rounding(plan, seed, call)
        for _ in range(calls):
            mode = w.pooling
            if w.nobag:
                assert opt == oracle.SGD
                E.emb_nobag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B,
                                    dw.grad_output, w.lr, E.EMB_NOBAG_AUTO, None)
            elif opt == oracle.SGD:
                E.emb_bag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B,
                                  dw.per_sample_weights, dw.grad_output, mode, w.lr, None)
            elif opt == oracle.ROWWISE_ADAGRAD:
                E.emb_bag_bwd_rowwise_adagrad(plan, dw.weights, mom, dw.indices, dw.offsets, w.N,
                                              w.B, dw.per_sample_weights, dw.grad_output, mode,
                                              w.lr, w.eps, None)
            else:
                E.emb_bag_bwd_adagrad(plan, dw.weights, mom, dw.indices, dw.offsets, w.N, w.B,
                                      dw.per_sample_weights, dw.grad_output, mode, w.lr, w.eps)
            assert E.emb_plan_status(plan) == E.EMB_OK
        state = E.emb_plan_get_rounding(plan)
    finally:
        E.emb_plan_destroy(plan)
    return dev.weights_numpy(dw), (None if mom is None else mom.cpu().numpy()), state


def oracle_update(w, opt, seed, call, m0=None, weights=None):
    """The oracle's step with stochastic rounding (seed, call), or round to nearest
    when seed is None."""
    exp = np.array(w.weights if weights is None else weights, copy=True)
    m = None if m0 is None else m0.copy()
    oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, exp,
                    w.indices, w.offsets, w.grad_output, optimizer=opt, lr=w.lr, eps=w.eps,
                    momentum=m, per_sample_weights=w.per_sample_weights,
                    mean=(w.pooling == synth.MEAN), nobag=w.nobag, grad_dtype=w.grad_dtype,
                    stochastic_rounding=None if seed is None else (seed, call))
    return exp, m


def check_sr_bits(w, opt, got, exp, w_old, m_old, mask, max_share=MAX_MISMATCH):
    """Touched elements: equal, one ulp apart, or further apart only within the
    derived bar of stochastic rounding (two spacings plus the a-priori bound of
    the device's fp32 update, tests/_bounds.py); few differ. Untouched:
    bit-identical."""
    gb, eb = got.view(np.uint16), exp.view(np.uint16)
    assert np.array_equal(gb[~mask], eb[~mask]), "untouched rows changed"
    d = ulp_diff16(gb[mask], eb[mask])
    check16(w, opt, got, exp, w_old, m_old, sr=True)
    assert (d != 0).mean() <= max_share, f"{(d != 0).sum()} of {d.size} elements differ"


def touched_mask(w):
    keys = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, 32)["run_keys"]
    mask = np.zeros(w.weights.size, bool)
    for k in keys:
        t = int(np.searchsorted(w.hash_size_cumsum, k, side="right") - 1)
        D = int(w.dims[t])
        o = int(w.weights_offsets[t]) + (int(k) - int(w.hash_size_cumsum[t])) * D
        mask[o:o + D] = True
    return mask


def check_parity(w, opt, seed=1234, call=7):
    m0 = state_init(w, opt)
    got, got_m, _ = gpu_update(w, opt, SR, seed, call, m0=m0)
    exp, exp_m = oracle_update(w, opt, seed, call, m0=m0)
    mask = touched_mask(w)
    check_sr_bits(w, opt, got, exp, w.weights, m0, mask)
    if got_m is not None:
        np.testing.assert_allclose(got_m, exp_m, rtol=1e-4, atol=1e-5)
    return got, mask


@pytest.mark.parametrize("wdt", [synth.F16, synth.BF16])
@pytest.mark.parametrize("opt", [oracle.SGD, oracle.ROWWISE_ADAGRAD, oracle.ADAGRAD])
def test_sr_parity(wdt, opt):
    w = custom(1, [300, 50, 2000], [8, 64, 20], 128, lambda r, T, B: r.integers(0, 30, (T, B)),
               weight_dtype=wdt, pooling=synth.MEAN, weighted=True, lr=0.05, eps=1e-4)
    check_parity(w, opt)


@pytest.mark.parametrize("wdt", [synth.F16, synth.BF16])
def test_sr_parity_dlrm_shape(wdt):
    w = synth.dlrm(5)
    w = custom(2, list(w.rows), list(w.dims), 512, lambda r, T, B: r.integers(0, 20, (T, B)),
               weight_dtype=wdt, lr=0.02)
    check_parity(w, oracle.SGD)


@pytest.mark.parametrize("D", [4, 260, 4096])
def test_sr_parity_row_widths_and_hot_rows(D):
    # chunked wide rows and hot rows split over warps keep the row-relative
    # vector index in the counter
    w = custom(3, [64, 33], [D, D], 64, lambda r, T, B: r.integers(0, 60, (T, B)),
               ids_fn=lambda r, t, n: np.where(r.random(n) < 0.5, 0, r.integers(0, 33, n)).astype(np.int64),
               weight_dtype=synth.BF16, lr=0.05)
    check_parity(w, oracle.SGD)


def test_sr_parity_unpooled():
    w = custom(4, [100, 3000, 17], [64, 64, 64], 4, lambda r, T, B: r.integers(0, 50, (T, B)),
               weight_dtype=synth.F16, nobag=True, lr=0.05)
    check_parity(w, oracle.SGD)


def test_sr_is_random_and_deterministic():
    w = custom(5, [500, 80], [32, 16], 256, lambda r, T, B: r.integers(0, 10, (T, B)),
               weight_dtype=synth.BF16, lr=0.05)
    mask = touched_mask(w)
    a, _, _ = gpu_update(w, oracle.SGD, SR, 99, 3)
    b, _, _ = gpu_update(w, oracle.SGD, SR, 99, 3)
    assert np.array_equal(a, b)  # same seed and call: same bits
    c, _, _ = gpu_update(w, oracle.SGD, SR, 99, 4)
    rn, _, _ = gpu_update(w, oracle.SGD, 0)
    for other in (c, rn):
        share = (a[mask] != other[mask]).mean()
        # rounding to the other neighbour than a second draw (or than the nearest)
        # happens for about a quarter to a half of the elements
        assert 0.1 < share < 0.6, share


def test_call_number_advances_per_update():
    w = custom(6, [400, 90], [32, 8], 64, lambda r, T, B: r.integers(0, 12, (T, B)),
               weight_dtype=synth.F16, lr=0.05)
    got, _, state = gpu_update(w, oracle.SGD, SR, 5, 11, calls=2)
    assert state == (5, 13)
    # the device's first call, then the second call from those weights
    first, _, _ = gpu_update(w, oracle.SGD, SR, 5, 11)
    exp, _ = oracle_update(w, oracle.SGD, 5, 12, weights=first)
    check_sr_bits(w, oracle.SGD, got, exp, first, None, touched_mask(w))


def test_sr_unbiased_on_device():
    # every touched element updates 1.0 - lr * 1.0 with lr = 0.3 * 2^-8: its bf16
    # neighbours are 1 - 2^-8 and 1.0, and the share of 1.0s must match the
    # dropped fraction of the fp32 update (low 16 bits / 2^16)
    rows, D, B = 2000, 128, 2000
    w = custom(7, [rows], [D], B, lambda r, T, B_: np.ones((T, B_), np.int64),
               ids_fn=lambda r, t, n: np.arange(n, dtype=np.int64), weight_dtype=synth.BF16,
               lr=0.3 * 2.0 ** -8)
    w.weights = np.full(w.weights.size, 0x3F80, np.uint16)  # 1.0
    w.grad_output = np.ones_like(w.grad_output)
    got, _, _ = gpu_update(w, oracle.SGD, SR, 2024, 0)
    n32 = np.float32(1.0) - np.float32(w.lr)
    frac = int(np.array([n32]).view(np.uint32)[0] & 0xFFFF) / 65536.0
    assert set(np.unique(got).tolist()) <= {0x3F80, 0x3F7F}
    share = (got == 0x3F80).mean()
    sigma = np.sqrt(frac * (1 - frac) / got.size)
    assert abs(share - frac) < 5 * sigma, (share, frac)


def test_fp32_weights_and_dense_mode_ignore_the_flag():
    w = custom(8, [300, 50], [16, 32], 64, lambda r, T, B: r.integers(0, 10, (T, B)), lr=0.05)
    a, _, sa = gpu_update(w, oracle.SGD, SR, 1, 0)
    b, _, _ = gpu_update(w, oracle.SGD, 0)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert sa == (1, 0)  # fp32 stores take no call number
    # the dense-gradient mode stores G, not an update: no stochastic rounding
    import torch
    wb = custom(9, [300, 50], [16, 32], 64, lambda r, T, B: r.integers(0, 10, (T, B)),
                weight_dtype=synth.BF16)
    dw = dev.to_device(wb)
    outs = []
    for flags in (SR, 0):
        buf = torch.empty(wb.weights.size, dtype=torch.bfloat16, device="cuda")
        plan = dev.make_plan(wb, flags=flags)
        try:
            E.emb_bag_bwd_dense_grad(plan, buf, dw.indices, dw.offsets, wb.N, wb.B, None,
                                     dw.grad_output, wb.pooling)
            assert E.emb_plan_status(plan) == E.EMB_OK
            assert E.emb_plan_get_rounding(plan) == (0, 0)
        finally:
            E.emb_plan_destroy(plan)
        outs.append(buf.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
