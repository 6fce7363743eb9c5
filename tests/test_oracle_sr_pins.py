"""Pins for the oracle's stochastic rounding against things other than itself.

* Philox4x32-10: the known-answer vectors published with the generator
  (counter and key all zero, all ones, and the digits-of-pi pair);
* bf16: over all 2^16 random words, the number of roundings away from zero
  equals the dropped low half of the fp32 pattern, exactly (an unbiased
  rounding); values already representable never move;
* fp16: over evenly spaced random words, the number of roundings away from zero
  matches the fraction (|x| - |lo|) / ulp computed independently with numpy's
  fp16 (the two neighbours of x);
* the backward with stochastic rounding stores, for every updated element, one of
  the two fp16 / bf16 values that bracket the update computed in fp32.
"""
import numpy as np
import pytest

from sparse_embedding_bag_gb300 import synth

MASK = 0xFFFFFFFF


def test_philox_known_answers(oracle_mod):
    kat = [
        ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
        ((MASK,) * 4, (MASK, MASK), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
        ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
         (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
    ]
    for ctr, key, exp in kat:
        assert oracle_mod.philox4x32_10(ctr, key).tolist() == list(exp)


def f32_bits(x):
    return int(np.array([x], np.float32).view(np.uint32)[0])


@pytest.mark.parametrize("x", [1.0 + 3.0 / 1024, -0.3, 123.456, 1e-30])
def test_sr_bf16_counts_equal_dropped_fraction(oracle_mod, x):
    u = f32_bits(x)
    lo = u >> 16
    low = u & 0xFFFF
    ups = 0
    for r in range(0, 1 << 16):
        b = oracle_mod.sr_bf16_bits(x, r)
        assert b in (lo, lo + 1)
        ups += b == lo + 1
    assert ups == low


def test_sr_bf16_representable_values_do_not_move(oracle_mod):
    for x in (1.0, -2.5, 0.0, 2.0 ** 127):
        u = f32_bits(x)
        assert u & 0xFFFF == 0
        for r in (0, 1, 0x7FFF, 0xFFFF, 0x12345678):
            assert oracle_mod.sr_bf16_bits(x, r) == u >> 16


@pytest.mark.parametrize("x", [1.0 + 1.0 / 3.0, -0.7, 1000.3, 3.0e-6, -6.1e-5])
def test_sr_half_counts_match_numpy_fraction(oracle_mod, x):
    xf = np.float32(x)
    near = np.float16(xf)
    lo = near if abs(float(near)) <= abs(float(xf)) else np.nextafter(near, np.float16(0))
    hi = np.nextafter(lo, np.float16(np.copysign(np.inf, float(xf))))
    frac = (abs(float(xf)) - abs(float(lo))) / (abs(float(hi)) - abs(float(lo)))
    thresh = frac * 2.0 ** 24  # an integer: both values are exact in fp32
    assert thresh == int(thresh)
    step = 1 << 12
    ups = 0
    lo_b, hi_b = int(np.array([lo]).view(np.uint16)[0]), int(np.array([hi]).view(np.uint16)[0])
    for k in range(0, 1 << 24, step):
        b = oracle_mod.sr_half_bits(float(xf), k << 8)
        assert b in (lo_b, hi_b)
        ups += b == hi_b
    assert ups == -(-int(thresh) // step)  # ceil(thresh / step)


def bracket16(v32, dtype):
    """Bit pattern of the fp16 / bf16 neighbour toward zero of the fp32 values v32
    (the one away from zero is that pattern plus one)."""
    if dtype == synth.F16:
        near = v32.astype(np.float16)
        over = np.abs(near.astype(np.float64)) > np.abs(v32.astype(np.float64))
        lo = np.where(over, np.nextafter(near, np.float16(0)), near)
        return lo.view(np.uint16).astype(np.int64), None
    u = v32.view(np.uint32).astype(np.int64)
    return u >> 16, None


@pytest.mark.parametrize("wdt", [synth.F16, synth.BF16])
def test_backward_sr_stores_a_bracketing_value(oracle_mod, wdt):
    rng = np.random.default_rng(5)
    rows, B = [60, 20], 40
    w = synth.make_bag_workload("sr", 5, rows, [8, 16], B, rng.integers(0, 6, (2, B)),
                                lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                weight_dtype=wdt, lr=0.03)
    keys, G = oracle_mod.row_grads(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.indices,
                                   w.offsets, w.grad_output)
    wd = (w.weights.astype(np.uint32) << 16).view(np.float32).astype(np.float64) \
        if wdt == synth.BF16 else w.weights.astype(np.float64)
    upd = wd.copy()
    for r, k in enumerate(keys):
        t = int(np.searchsorted(w.hash_size_cumsum, k, side="right") - 1)
        D = int(w.dims[t])
        o = int(w.weights_offsets[t]) + (int(k) - int(w.hash_size_cumsum[t])) * D
        upd[o:o + D] = wd[o:o + D] - np.float64(np.float32(0.03)) * G[r, :D]
    got = np.array(w.weights, copy=True)
    oracle_mod.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, got,
                        w.indices, w.offsets, w.grad_output, optimizer=oracle_mod.SGD, lr=0.03,
                        stochastic_rounding=(1234, 7))
    lo, _ = bracket16(upd.astype(np.float32), wdt)
    gb = got.view(np.uint16).astype(np.int64)
    # one of the two neighbours (toward / away from zero) of the fp32 update
    assert np.all((gb == lo) | (gb == lo + 1))
    # and it is random: with another call number some element rounds the other way
    got2 = np.array(w.weights, copy=True)
    oracle_mod.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, got2,
                        w.indices, w.offsets, w.grad_output, optimizer=oracle_mod.SGD, lr=0.03,
                        stochastic_rounding=(1234, 8))
    assert not np.array_equal(got, got2)


def test_sr_half_saturates_and_passes_inf(oracle_mod):
    # beyond the largest finite fp16 (65504 = 0x7BFF) the neighbour away from zero
    # would be infinity: the update stays at the largest finite value
    for r in (0, 1 << 8, 0xFFFFFF00):
        assert oracle_mod.sr_half_bits(70000.0, r) == 0x7BFF
        assert oracle_mod.sr_half_bits(-1e9, r) == 0xFBFF
        assert oracle_mod.sr_half_bits(65504.0, r) == 0x7BFF
        assert oracle_mod.sr_half_bits(float("inf"), r) == 0x7C00
        assert oracle_mod.sr_half_bits(float("-inf"), r) == 0xFC00
    # just below 65504 the rule still rounds up with the dropped fraction
    assert oracle_mod.sr_half_bits(65500.0, 0) == 0x7BFF  # (65500 - 65472) / 32 > 0: r = 0 rounds up
    assert oracle_mod.sr_half_bits(65500.0, 0xFFFFFF00) == 0x7BFE
