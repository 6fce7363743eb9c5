"""Pins for the CPU oracle against things other than itself.

* hand-worked examples (tests/golden/*.json, exact dyadic arithmetic);
* brute force: the row gradient as a dense one-hot matrix product A_t^T g_t
  (numpy matmul), for sum / mean / weighted / unpooled lookups;
* brute-force integer outputs (Python dict counting);
* invariants: gradient-sum identities, linearity, bag-permutation invariance;
* closed forms of one SGD / row-wise Adagrad step;
* the storage conversions against numpy (fp16), torch (bf16 from fp32-exact
  values) and textbook round-to-nearest-even tie cases.
"""
import json
import math
import os

import numpy as np
import pytest

from sparse_embedding_bag_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bag_tables(w):
    """(t, b, i) for every lookup, straight from the CSR."""
    out = []
    for bt in range(w.T * w.B):
        t, b = divmod(bt, w.B)
        for i in range(int(w.offsets[bt]), int(w.offsets[bt + 1])):
            out.append((t, b, i))
    return out


def brute_force_G(w, psw=None, mean=False, nobag=False):
    """Dense one-hot A_t[b, r] (or [l, r] unpooled) and G_t = A_t^T g_t for every table."""
    Gs = {}
    g_all = w.grad_output.astype(np.float64)
    for t in range(w.T):
        E, D = int(w.rows[t]), int(w.dims[t])
        if nobag:
            A = np.zeros((w.N, E))
            g = g_all
        else:
            A = np.zeros((w.B, E))
            g = g_all[:, int(w.D_offsets[t]):int(w.D_offsets[t + 1])]
        for bt in range(t * w.B, (t + 1) * w.B):
            b = bt - t * w.B
            L = int(w.offsets[bt + 1] - w.offsets[bt])
            for i in range(int(w.offsets[bt]), int(w.offsets[bt + 1])):
                s = 1.0 if psw is None else float(psw[i])
                if mean:
                    s /= L
                A[i if nobag else b, int(w.indices[i])] += s
        touched = np.zeros(E, bool)
        for bt in range(t * w.B, (t + 1) * w.B):
            touched[w.indices[int(w.offsets[bt]):int(w.offsets[bt + 1])]] = True
        Gt = A.T @ g
        Gs[t] = (touched, Gt)
        assert Gt.shape == (E, D)
    return Gs


def check_against_brute(oracle_mod, w, psw=None, mean=False, nobag=False, rtol=1e-12):
    keys, G = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices,
                                   w.offsets, w.grad_output, per_sample_weights=psw, mean=mean,
                                   nobag=nobag)
    Gs = brute_force_G(w, psw, mean, nobag)
    hsc = w.hash_size_cumsum
    expect_keys = []
    for t in range(w.T):
        touched, _ = Gs[t]
        expect_keys.extend(int(hsc[t]) + np.nonzero(touched)[0])
    np.testing.assert_array_equal(keys, np.array(expect_keys, np.int64))
    for r, k in enumerate(keys):
        t = int(np.searchsorted(hsc, k, side="right") - 1)
        D = int(w.dims[t])
        np.testing.assert_allclose(G[r, :D], Gs[t][1][k - hsc[t]], rtol=rtol, atol=1e-12)
        assert np.all(G[r, D:] == 0)


def small_workload(seed, T=3, B=7, rows=(5, 9, 3), dims=(4, 8, 12), maxlen=6, nobag=False):
    rng = np.random.default_rng(seed + 100)
    if nobag:
        dims = (dims[0],) * T
    lengths = rng.integers(0, maxlen + 1, size=(T, B))
    return synth.make_bag_workload("small", seed, list(rows)[:T], list(dims)[:T], B, lengths,
                                   lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                   weighted=True, nobag=nobag)


# ---------------------------------------------------------------- hand examples

def test_hand_runs(oracle_mod):
    h = _load("hand_pooled.json")
    keys, ids = oracle_mod.sorted_pairs(h["T"], h["B"], h["hash_size_cumsum"], h["indices"],
                                        h["offsets"])
    assert ids.tolist() == h["runs"]["sorted_ids"]
    r = oracle_mod.runs(h["T"], h["B"], h["hash_size_cumsum"], h["indices"], h["offsets"], 2)
    assert r["run_keys"].tolist() == h["runs"]["run_keys"]
    assert r["run_len"].tolist() == h["runs"]["run_len"]
    assert r["cum"].tolist() == h["runs"]["cum"]
    assert r["long_ids"].tolist() == h["runs"]["long_ids_thr2"]


@pytest.mark.parametrize("variant", ["sum", "mean", "sum_weighted"])
def test_hand_row_grads(oracle_mod, variant):
    h = _load("hand_pooled.json")
    g = np.array(h["grad_output"], np.float32)
    psw = np.array(h["per_sample_weights"], np.float32) if variant == "sum_weighted" else None
    keys, G = oracle_mod.row_grads(h["T"], h["B"], h["hash_size_cumsum"], h["D_offsets"],
                                   h["indices"], h["offsets"], g, per_sample_weights=psw,
                                   mean=(variant == "mean"))
    expect = h["G_" + variant]
    assert [str(k) for k in keys] == list(expect.keys())
    for r, k in enumerate(keys):
        assert G[r].tolist() == expect[str(k)]  # exact: dyadic arithmetic


@pytest.mark.parametrize("wdtype", [np.float32, np.float16])
def test_hand_sgd(oracle_mod, wdtype):
    h = _load("hand_pooled.json")
    g = np.array(h["grad_output"], np.float32)
    w = np.full(20, h["sgd_w0"], wdtype)
    oracle_mod.backward(h["T"], h["B"], h["hash_size_cumsum"], h["D_offsets"],
                        h["weights_offsets"], w, h["indices"], h["offsets"], g,
                        optimizer=oracle_mod.SGD, lr=h["sgd_lr"])
    assert w.astype(np.float64).tolist() == h["sgd_sum_weights_after"]


def test_hand_adagrad(oracle_mod):
    h = _load("hand_adagrad.json")
    g = np.array(h["grad_output"], np.float32)
    w = np.array(h["weights_in"], np.float32)
    m = np.array(h["momentum_in"], np.float32)
    keys, G = oracle_mod.row_grads(h["T"], h["B"], h["hash_size_cumsum"], h["D_offsets"],
                                   h["indices"], h["offsets"], g)
    for r, k in enumerate(keys):
        assert G[r].tolist() == h["G"][str(k)]
    oracle_mod.backward(h["T"], h["B"], h["hash_size_cumsum"], h["D_offsets"],
                        h["weights_offsets"], w, h["indices"], h["offsets"], g,
                        optimizer=oracle_mod.ROWWISE_ADAGRAD, lr=h["lr"], eps=h["eps"],
                        momentum=m)
    assert m.tolist() == h["momentum_out"]
    rows_023 = np.concatenate([w[0:4], w[8:12], w[12:16]])
    assert rows_023.astype(np.float64).tolist() == h["weights_out_rows_0_2_3"]
    # row 1: m = 20, sqrt(20) is irrational; closed form in double, rounded once to fp32
    exp = [np.float32(2.0 - 0.5 * gd / math.sqrt(20.0)) for gd in (0, 4, 4, 0)]
    assert w[4:8].tolist() == [float(x) for x in exp]


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", ["sum", "mean", "weighted", "weighted_mean"])
def test_row_grads_vs_one_hot_matmul(oracle_mod, seed, mode):
    w = small_workload(seed)
    psw = w.per_sample_weights if "weighted" in mode else None
    check_against_brute(oracle_mod, w, psw=psw, mean=("mean" in mode))


@pytest.mark.parametrize("seed", [0, 1])
def test_row_grads_nobag_vs_one_hot_matmul(oracle_mod, seed):
    w = small_workload(seed, nobag=True)
    check_against_brute(oracle_mod, w, nobag=True)


def test_row_grads_tiny_config_vs_one_hot(oracle_mod):
    check_against_brute(oracle_mod, synth.tiny(0))


def test_row_grads_bf16_grad_vs_one_hot(oracle_mod):
    w = small_workload(3, nobag=True)
    import torch
    bits = torch.from_numpy(w.grad_output).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    exact = torch.from_numpy(w.grad_output).to(torch.bfloat16).to(torch.float64).numpy()
    keys, G = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices,
                                   w.offsets, bits, nobag=True)
    w2 = small_workload(3, nobag=True)
    w2.grad_output = exact
    Gs = brute_force_G(w2, nobag=True)
    for r, k in enumerate(keys):
        t = int(np.searchsorted(w.hash_size_cumsum, k, side="right") - 1)
        np.testing.assert_allclose(G[r, :w.dims[t]], Gs[t][1][k - w.hash_size_cumsum[t]],
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- integer outputs

@pytest.mark.parametrize("seed", [0, 5])
@pytest.mark.parametrize("thr", [1, 2, 3, 32])
def test_runs_vs_counting(oracle_mod, seed, thr):
    w = small_workload(seed, maxlen=9)
    counts = {}
    for t, b, i in _bag_tables(w):
        k = int(w.hash_size_cumsum[t] + w.indices[i])
        counts[k] = counts.get(k, 0) + 1
    keys = sorted(counts)
    r = oracle_mod.runs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets, thr)
    assert r["run_keys"].tolist() == keys
    assert r["run_len"].tolist() == [counts[k] for k in keys]
    assert r["num_runs"] == len(keys)
    assert int(r["run_len"].sum()) == w.N
    assert r["cum"][0] == 0 and r["cum"][-1] == w.N
    assert np.all(np.diff(r["cum"]) == r["run_len"])
    assert r["long_ids"].tolist() == [j for j, k in enumerate(keys) if counts[k] >= thr]


def test_sorted_pairs_stable_ties(oracle_mod):
    w = small_workload(7, maxlen=9)
    keys, ids = oracle_mod.sorted_pairs(w.T, w.B, w.hash_size_cumsum, w.indices, w.offsets)
    assert np.all(np.diff(keys) >= 0)
    same = np.diff(keys) == 0
    assert np.all(np.diff(ids)[same] > 0)  # ties in lookup-id order
    assert sorted(ids.tolist()) == list(range(w.N))


def test_empty_and_error_codes(oracle_mod):
    r = oracle_mod.runs(1, 2, [0, 10], np.zeros(0, np.int64), [0, 0, 0], 32)
    assert r["num_runs"] == 0 and r["cum"].tolist() == [0]
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.runs(1, 1, [0, 10], [3, 10], [0, 2], 32)
    assert e.value.code == 3
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.runs(1, 1, [0, 10], [3, -1], [0, 2], 32)
    assert e.value.code == 3
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.runs(1, 2, [0, 10], [3, 1], [0, 2, 1], 32)  # offsets decrease
    assert e.value.code == 1


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("mode", ["sum", "weighted", "mean"])
def test_gradient_sum_invariant(oracle_mod, mode):
    w = small_workload(11, maxlen=8)
    psw = w.per_sample_weights if mode == "weighted" else None
    keys, G = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices,
                                   w.offsets, w.grad_output, per_sample_weights=psw,
                                   mean=(mode == "mean"))
    for t in range(w.T):
        D = int(w.dims[t])
        sel = (keys >= w.hash_size_cumsum[t]) & (keys < w.hash_size_cumsum[t + 1])
        lhs = G[sel, :D].sum(axis=0)
        g = w.grad_output[:, w.D_offsets[t]:w.D_offsets[t + 1]].astype(np.float64)
        rhs = np.zeros(D)
        for b in range(w.B):
            bt = t * w.B + b
            a, e = int(w.offsets[bt]), int(w.offsets[bt + 1])
            if mode == "sum":
                coef = e - a
            elif mode == "weighted":
                coef = float(psw[a:e].astype(np.float64).sum())
            else:
                coef = 1.0 if e > a else 0.0
            rhs += coef * g[b]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-10)


def test_linearity_and_bag_permutation(oracle_mod):
    w = small_workload(13, maxlen=5)
    rng = np.random.default_rng(99)
    g1 = w.grad_output
    g2 = rng.standard_normal(g1.shape).astype(np.float32)
    args = (w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices, w.offsets)
    k1, G1 = oracle_mod.row_grads(*args, g1)
    _, G2 = oracle_mod.row_grads(*args, g2)
    # 2*g1 and g1+g2 are exact in fp32 only approximately; compare in double tolerance
    k3, G3 = oracle_mod.row_grads(*args, (2.0 * g1).astype(np.float32))
    np.testing.assert_allclose(G3, 2.0 * G1, rtol=1e-12)
    # permute the bags of every table together with their grad rows
    perm = rng.permutation(w.B)
    new_off = [0]
    new_idx = []
    for t in range(w.T):
        for b in range(w.B):
            bt = t * w.B + perm[b]
            seg = w.indices[int(w.offsets[bt]):int(w.offsets[bt + 1])]
            new_idx.extend(seg.tolist())
            new_off.append(new_off[-1] + len(seg))
    g_perm = g1[perm]
    k4, G4 = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets,
                                  np.array(new_idx, np.int64), np.array(new_off, np.int64), g_perm)
    np.testing.assert_array_equal(k4, k1)
    np.testing.assert_allclose(G4, G1, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_sgd_single_lookup_closed_form(oracle_mod):
    w = np.array([0.5, -0.25, 1.0, 2.0, 7.0, 7.0, 7.0, 7.0], np.float32)
    g = np.array([[3.0, -1.0, 0.5, 4.0]], np.float32)
    oracle_mod.backward(2, 1, [0, 1, 2], [0, 4, 8], [0, 4], w, [0], [0, 1, 1],
                        np.concatenate([g, g], axis=1), optimizer=oracle_mod.SGD, lr=0.25)
    assert w[:4].tolist() == [0.5 - 0.75, -0.25 + 0.25, 1.0 - 0.125, 2.0 - 1.0]
    assert w[4:].tolist() == [7.0] * 4  # untouched table


@pytest.mark.parametrize("D", [4, 16, 64, 256, 1028, 2048, 4096])
def test_adagrad_from_zero_closed_form(oracle_mod, D):
    # (1028-4096: rows the device updates in two launches, its state from the sums
    # of squares of 1024-wide chunks)
    rng = np.random.default_rng(D)
    g = rng.standard_normal((1, D)).astype(np.float32)
    w = rng.uniform(-1, 1, D).astype(np.float32)
    w0 = w.copy()
    m = np.zeros(1, np.float32)
    lr, eps = float(np.float32(0.01)), float(np.float32(1e-8))
    oracle_mod.backward(1, 1, [0, 1], [0, D], [0], w, [0], [0, 1], g,
                        optimizer=oracle_mod.ROWWISE_ADAGRAD, lr=lr, eps=eps, momentum=m)
    gd = g[0].astype(np.float64)
    rms = math.sqrt(float((gd * gd).mean()))
    assert m[0] == np.float32(rms * rms)
    step = np.linalg.norm(w.astype(np.float64) - w0.astype(np.float64))
    expect = lr * np.linalg.norm(gd) / (rms + eps)
    assert abs(step - expect) <= 1e-6 * expect
    assert abs(expect - lr * math.sqrt(D)) <= 1e-5 * expect  # ||G|| / rms(G) = sqrt(D)


def test_untouched_rows_bit_identical(oracle_mod):
    w = synth.dlrm(0)
    # shrink: first 64 bags of each table
    B = 64
    offs = [0]
    idx = []
    for t in range(w.T):
        for b in range(B):
            bt = t * w.B + b
            seg = w.indices[int(w.offsets[bt]):int(w.offsets[bt + 1])]
            idx.extend(seg.tolist())
            offs.append(offs[-1] + len(seg))
    idx = np.array(idx, np.int64)
    offs = np.array(offs, np.int64)
    g = w.grad_output[:B]
    weights = w.weights.copy()
    m = w.momentum.copy()
    oracle_mod.backward(w.T, B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, weights, idx,
                        offs, g, optimizer=oracle_mod.ROWWISE_ADAGRAD, lr=w.lr, eps=w.eps,
                        momentum=m)
    touched = np.zeros(int(w.hash_size_cumsum[-1]), bool)
    for t in range(w.T):
        seg = idx[offs[t * B]:offs[(t + 1) * B]]
        touched[w.hash_size_cumsum[t] + seg] = True
    rows_w = weights.reshape(-1, 64)
    rows_w0 = w.weights.reshape(-1, 64)
    assert np.array_equal(rows_w[~touched].view(np.uint32), rows_w0[~touched].view(np.uint32))
    assert np.all(m[~touched] == 0) and np.all(m[touched] > 0)
    assert np.all(np.any(rows_w[touched] != rows_w0[touched], axis=1))


# ---------------------------------------------------------------- conversions

def test_half_conversion_vs_numpy(oracle_mod):
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000),
                         [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -24, 2.0 ** -25,
                          3 * 2.0 ** -26, 2.0 ** -14 - 2.0 ** -26, np.inf, -np.inf, 1e300, -1e300]])
    for x in xs:
        assert oracle_mod.double_to_half_bits(x) == int(np.float64(x).astype(np.float16).view(np.uint16)), x
    for h in range(0, 0x7C00, 37):
        assert oracle_mod.half_bits_to_double(h) == float(np.uint16(h).view(np.float16))


def test_half_ties_to_even(oracle_mod):
    assert oracle_mod.double_to_half_bits(1.0 + 2.0 ** -11) == 0x3C00  # tie -> even (down)
    assert oracle_mod.double_to_half_bits(1.0 + 3 * 2.0 ** -11) == 0x3C02  # tie -> even (up)
    assert oracle_mod.double_to_half_bits(1.0 + 2.0 ** -11 + 2.0 ** -40) == 0x3C01  # above tie


def test_bf16_conversion(oracle_mod):
    import torch
    rng = np.random.default_rng(1)
    xs = np.concatenate([(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)),
                         [np.inf, -np.inf, 3.4e38, -3.4e38]]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, r in zip(xs, ref):
        assert oracle_mod.double_to_bf16_bits(float(x)) == int(r), x
    assert oracle_mod.double_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80  # tie -> even
    assert oracle_mod.double_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above a tie: direct rounding goes up (rounding via fp32 first would not)
    assert oracle_mod.double_to_bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    for h in range(0, 0x7F80, 97):
        assert oracle_mod.bf16_bits_to_double(h) == float(
            torch.tensor([h], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float())


def test_adagrad_eps_outside_sqrt(oracle_mod):
    """lr=3, eps=2 on the hand example: rows 0 and 2 have sqrt(m')=2 and 4, so
    w' = w - 3*G/(sqrt(m')+2) is dyadic; eps inside the root (or the old state)
    would give irrational values."""
    h = _load("hand_adagrad.json")
    g = np.array(h["grad_output"], np.float32)
    w = np.array(h["weights_in"], np.float32)
    m = np.array(h["momentum_in"], np.float32)
    oracle_mod.backward(h["T"], h["B"], h["hash_size_cumsum"], h["D_offsets"],
                        h["weights_offsets"], w, h["indices"], h["offsets"], g,
                        optimizer=oracle_mod.ROWWISE_ADAGRAD, lr=3.0, eps=2.0, momentum=m)
    assert w[0:4].tolist() == [2.5, -0.5, -0.5, 2.5]   # 1 - 3*G/(2+2)
    assert w[8:12].tolist() == [5.0, 3.0, 3.0, 5.0]    # 4 - 3*G/(4+2)
    assert m.tolist() == h["momentum_out"]
