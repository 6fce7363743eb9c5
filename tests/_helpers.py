"""Shared helpers of the GPU parity tests: run a workload through the C ABI and
compare with the CPU oracle (element by element on the same seeded inputs)."""
import numpy as np

import oracle
from sparse_embedding_bag_gb300 import device as dev
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import synth

RTOL, ATOL = 1e-4, 1e-5  # fp32 weights and momentum
# fp16 / bf16 weights: at most 1 ulp from the oracle's rounded value, or, where the
# update cancels, within one spacing plus the a-priori bound of the device's fp32
# arithmetic (tests/_bounds.py)
MAX_ULP = 1


def ordered_bits16(bits: np.ndarray) -> np.ndarray:
    """Maps fp16/bf16 bit patterns to integers whose difference counts ulps."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_diff16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordered_bits16(a_bits) - ordered_bits16(b_bits))


def oracle_step(w: synth.Workload):
    """Oracle result (weights, momentum) of one step on host copies of w's inputs."""
    weights = np.array(w.weights, copy=True)
    momentum = None if w.momentum is None else np.array(w.momentum, copy=True)
    oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, weights,
                    w.indices, w.offsets, w.grad_output, optimizer=w.optimizer, lr=w.lr,
                    eps=w.eps, momentum=momentum, momentum_offsets=w.momentum_offsets,
                    per_sample_weights=w.per_sample_weights, mean=(w.pooling == synth.MEAN),
                    nobag=w.nobag, grad_dtype=w.grad_dtype)
    return weights, momentum


def compare_weights(w: synth.Workload, got: np.ndarray, exp: np.ndarray, touched_keys,
                    opt=None, w_old=None, m_old=None):
    """Touched rows within tolerance; untouched rows bit-identical. For 16-bit
    weights the tolerance is one ulp, or the derived bound where an update cancels
    (opt, w_old, m_old: the step's optimizer and the state before it; default
    the workload's)."""
    hsc = w.hash_size_cumsum
    keys = np.asarray(touched_keys, np.int64)
    for t in range(w.T):
        E_t, D = int(w.rows[t]), int(w.dims[t])
        o = int(w.weights_offsets[t])
        g2 = got[o:o + E_t * D].reshape(E_t, D)
        e2 = exp[o:o + E_t * D].reshape(E_t, D)
        idx = keys[(keys >= hsc[t]) & (keys < hsc[t + 1])] - hsc[t]
        mask = np.zeros(E_t, bool)
        mask[idx] = True
        if got.dtype == np.float32:
            np.testing.assert_allclose(g2[mask], e2[mask], rtol=RTOL, atol=ATOL,
                                       err_msg=f"table {t} touched rows")
            same = np.array_equal(g2[~mask].view(np.uint32), e2[~mask].view(np.uint32))
        else:
            same = np.array_equal(g2[~mask].view(np.uint16), e2[~mask].view(np.uint16))
        assert same, f"table {t}: untouched rows changed"
    if got.dtype != np.float32:
        from _bounds import check16
        check16(w, w.optimizer if opt is None else opt, got, exp,
                w.weights if w_old is None else w_old, w.momentum if m_old is None else m_old)


def compare_momentum(w: synth.Workload, got: np.ndarray, exp: np.ndarray):
    np.testing.assert_allclose(got, exp, rtol=RTOL, atol=ATOL)
    untouched = exp == w.momentum
    assert np.array_equal(got[untouched], exp[untouched])


def compare_runs(got: dict, exp: dict):
    """Integer outputs: bit-exact; long-run ids as a set."""
    assert got["num_runs"] == exp["num_runs"]
    np.testing.assert_array_equal(got["run_keys"], exp["run_keys"])
    np.testing.assert_array_equal(got["run_len"], exp["run_len"])
    np.testing.assert_array_equal(got["cum"], exp["cum"])
    assert sorted(got["long_ids"].tolist()) == exp["long_ids"].tolist()


def run_and_check(w: synth.Workload, path=E.EMB_NOBAG_AUTO, thr=0, check_runs=True, plan_kw=None):
    """One step on the GPU through the C ABI, checked against the oracle. Returns the device workload."""
    dw = dev.to_device(w)
    plan = dev.make_plan(w, max_segment_length_per_warp=thr, **(plan_kw or {}))
    try:
        dev.step(plan, dw, path=path)
        assert E.emb_plan_status(plan) == E.EMB_OK
        sorted_path = not (w.nobag and path == E.EMB_NOBAG_ATOMIC)
        if check_runs and sorted_path:
            got = E.emb_plan_debug_runs(plan, max(w.N, 1))
            exp = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, thr or 32)
            compare_runs(got, exp)
    finally:
        E.emb_plan_destroy(plan)
    ew, em = oracle_step(w)
    touched = oracle.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, 32)["run_keys"]
    compare_weights(w, dev.weights_numpy(dw), ew, touched)
    if em is not None:
        compare_momentum(w, dw.momentum.cpu().numpy(), em)
    return dw
