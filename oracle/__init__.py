"""CPU oracle for the embedding backward pass with a fused row optimizer.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``sparse_embedding_bag_gb300``) never imports it
and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++, doubles
throughout, std::sort for the grouping); this module only builds it with g++
and marshals numpy arrays through ctypes. What each function follows:

* ``sorted_pairs`` / ``runs``: linearisation ``hash_size_cumsum[t] + idx`` and
  the sorted, run-length encoded lookup list with its long-run set
  ("fbgemm_gpu/codegen/embedding_backward_split_template.cu",
  ``*_find_long_segments`` and the per-row kernels' run bookkeeping).
* ``row_grads``: the de-duplicated per-row gradient, scaled per lookup by the
  per-sample weight and by 1/L under mean pooling (same page,
  ``grad_mean_kernel`` and the weighted accumulation in the per-row kernels).
* ``backward``: the row gradient followed by SGD or row-wise Adagrad once per
  unique row ("tt_embeddings_cuda.cu", ``update_tt_cores_sgd_kernel``,
  ``cache_backward_rowwise_adagrad_approx_kernel``), rounded to the weight's
  storage type with round-to-nearest-even.

Every function is pinned by ``tests/test_oracle_pins.py``. No expected value
in the test-suite is produced by the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
SGD, ROWWISE_ADAGRAD, ADAGRAD = 0, 1, 2
SUM, MEAN = 0, 1

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "index out of range"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned {code} ({_STATUS.get(code, '?')})")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (g++, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_sorted_pairs.argtypes = [i32, i32, vp, vp, vp, i64, vp, vp]
            lib.oracle_runs.argtypes = [i32, i32, vp, vp, vp, i64, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_row_grads.argtypes = [i32, i32, vp, vp, vp, vp, i64, vp, i32, i32, i32, vp,
                                             i32, vp, vp, vp]
            lib.oracle_apply_row.argtypes = [i32, i32, vp, i64, i32, vp, vp, f64, f64]
            lib.oracle_backward.argtypes = [i32, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, i64, vp,
                                            i32, i32, i32, vp, i32, f64, f64, i32, ctypes.c_uint64,
                                            ctypes.c_uint64]
            lib.oracle_philox4x32_10.argtypes = [vp, vp, vp]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_sr_bf16.argtypes = [ctypes.c_float, ctypes.c_uint32]
            lib.oracle_sr_bf16.restype = ctypes.c_uint16
            lib.oracle_sr_half.argtypes = [ctypes.c_float, ctypes.c_uint32]
            lib.oracle_sr_half.restype = ctypes.c_uint16
            lib.oracle_forward.argtypes = [i32, i32, vp, vp, vp, i32, vp, vp, vp, i64, vp, i32,
                                           i32, vp]
            lib.oracle_dense_grad.argtypes = [i32, i32, vp, vp, vp, i64, i32, vp, vp, vp, i64, vp,
                                              i32, i32, i32, vp]
            lib.oracle_bucketize.argtypes = [i32, i32, i32, vp, i32, vp, vp, i64, vp, i32, vp, vp,
                                             vp, vp]
            lib.oracle_merge.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp]
            for name in ("oracle_sorted_pairs", "oracle_runs", "oracle_row_grads",
                         "oracle_apply_row", "oracle_backward", "oracle_forward",
                         "oracle_dense_grad", "oracle_bucketize", "oracle_merge"):
                getattr(lib, name).restype = ctypes.c_int
            lib.oracle_double_to_half.argtypes = [f64]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = f64
            lib.oracle_double_to_bf16.argtypes = [f64]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = f64
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(code):
    if code != 0:
        raise OracleError(code)


def dtype_code(arr: np.ndarray, bf16: bool = False) -> int:
    """Storage code of a weight/grad array: fp32, fp16, or bf16 held as uint16 bits."""
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.float16:
        return F16
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"unsupported storage dtype {arr.dtype}")


def sorted_pairs(T, B, hash_size_cumsum, indices, offsets):
    hsc, idx, off = _c(hash_size_cumsum, np.int64), _c(indices, np.int64), _c(offsets, np.int64)
    N = idx.size
    keys = np.empty(N, np.int64)
    ids = np.empty(N, np.int64)
    _check(_load().oracle_sorted_pairs(T, B, _p(hsc), _p(idx), _p(off), N, _p(keys), _p(ids)))
    return keys, ids


def runs(T, B, hash_size_cumsum, indices, offsets, max_segment_length_per_warp=32):
    """Sorted unique linear indices, run lengths, cumulative run lengths, long run ids."""
    hsc, idx, off = _c(hash_size_cumsum, np.int64), _c(indices, np.int64), _c(offsets, np.int64)
    N = idx.size
    run_keys = np.empty(max(N, 1), np.int64)
    run_len = np.empty(max(N, 1), np.int32)
    cum = np.empty(N + 1, np.int32)
    long_ids = np.empty(max(N, 1), np.int32)
    U = ctypes.c_int64(0)
    nl = ctypes.c_int64(0)
    _check(_load().oracle_runs(T, B, _p(hsc), _p(idx), _p(off), N, max_segment_length_per_warp,
                               _p(run_keys), _p(run_len), _p(cum), ctypes.byref(U), _p(long_ids),
                               ctypes.byref(nl)))
    u = U.value
    return {"run_keys": run_keys[:u].copy(), "run_len": run_len[:u].copy(),
            "cum": cum[:u + 1].copy(), "num_runs": u, "long_ids": long_ids[:nl.value].copy()}


def row_grads(T, B, hash_size_cumsum, D_offsets, indices, offsets, grad_output, *,
              per_sample_weights=None, mean=False, nobag=False, grad_dtype=None):
    """De-duplicated row gradients (double): (keys[U], G[U, Dmax])."""
    hsc, Do = _c(hash_size_cumsum, np.int64), _c(D_offsets, np.int32)
    idx, off = _c(indices, np.int64), _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    g = np.ascontiguousarray(grad_output)
    gcode = dtype_code(g) if grad_dtype is None else grad_dtype
    N = idx.size
    Dmax = int(np.max(np.diff(Do)))
    keys = np.empty(max(N, 1), np.int64)
    G = np.zeros((max(N, 1), Dmax), np.float64)
    U = ctypes.c_int64(0)
    _check(_load().oracle_row_grads(T, B, _p(hsc), _p(Do), _p(idx), _p(off), N, _p(psw),
                                    int(bool(mean)), int(bool(nobag)), gcode, _p(g), Dmax,
                                    _p(keys), _p(G), ctypes.byref(U)))
    u = U.value
    return keys[:u].copy(), G[:u].copy()


def apply_row(optimizer, weights, row_offset, D, g, momentum=None, momentum_index=0,
              lr=0.01, eps=1e-8):
    """Optimizer step on one row of `weights` (in place); returns the new momentum (or None)."""
    code = dtype_code(weights)
    gd = np.ascontiguousarray(g, np.float64)
    m = None
    if optimizer == ROWWISE_ADAGRAD:
        m = np.array([momentum[momentum_index]], np.float32)
    elif optimizer == ADAGRAD:
        m = np.array(momentum[momentum_index:momentum_index + D], np.float32)
    _check(_load().oracle_apply_row(optimizer, code, _p(weights), row_offset, D, _p(gd), _p(m),
                                    float(lr), float(eps)))
    if optimizer == ADAGRAD:
        momentum[momentum_index:momentum_index + D] = m
        return m
    if m is not None:
        momentum[momentum_index] = m[0]
        return m[0]
    return None


def backward(T, B, hash_size_cumsum, D_offsets, weights_offsets, weights, indices, offsets,
             grad_output, *, optimizer, lr, eps=0.0, momentum=None, momentum_offsets=None,
             per_sample_weights=None, mean=False, nobag=False, grad_dtype=None,
             stochastic_rounding=None):
    """Full backward + in-place optimizer on numpy `weights` (and `momentum`).

    `weights` is float32, float16, or uint16 holding bfloat16 bits; `lr` and
    `eps` should be the exact fp32 values the device path receives.
    stochastic_rounding: None (round to nearest even) or (seed, call) for
    stochastic rounding of fp16 / bf16 weight stores.
    """
    hsc, Do = _c(hash_size_cumsum, np.int64), _c(D_offsets, np.int32)
    wo, mo = _c(weights_offsets, np.int64), _c(momentum_offsets, np.int64)
    idx, off = _c(indices, np.int64), _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    g = np.ascontiguousarray(grad_output)
    gcode = dtype_code(g) if grad_dtype is None else grad_dtype
    assert weights.flags.c_contiguous
    if momentum is not None:
        assert momentum.dtype == np.float32 and momentum.flags.c_contiguous
    _check(_load().oracle_backward(T, B, _p(hsc), _p(Do), _p(wo), _p(mo), dtype_code(weights),
                                   _p(weights), _p(momentum), _p(idx), _p(off), idx.size, _p(psw),
                                   int(bool(mean)), int(bool(nobag)), gcode, _p(g), optimizer,
                                   float(lr), float(eps), int(stochastic_rounding is not None),
                                   *(stochastic_rounding or (0, 0))))


def dense_grad(T, B, hash_size_cumsum, D_offsets, weights_offsets, extent, indices, offsets,
               grad_output, *, out_dtype=F32, per_sample_weights=None, mean=False, nobag=False,
               grad_dtype=None):
    """Dense-gradient mode: [extent] buffer (weights layout) of out_dtype, zero except the
    de-duplicated row gradients of the touched rows."""
    hsc, Do = _c(hash_size_cumsum, np.int64), _c(D_offsets, np.int32)
    wo = _c(weights_offsets, np.int64)
    idx, off = _c(indices, np.int64), _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    g = np.ascontiguousarray(grad_output)
    gcode = dtype_code(g) if grad_dtype is None else grad_dtype
    out = np.empty(int(extent), {F32: np.float32, F16: np.float16, BF16: np.uint16}[out_dtype])
    _check(_load().oracle_dense_grad(T, B, _p(hsc), _p(Do), _p(wo), int(extent), out_dtype,
                                     _p(out), _p(idx), _p(off), idx.size, _p(psw), int(bool(mean)),
                                     int(bool(nobag)), gcode, _p(g)))
    return out


def forward(T, B, hash_size_cumsum, D_offsets, weights_offsets, weights, indices, offsets, *,
            per_sample_weights=None, mean=False, out_dtype=F32):
    """Forward pooled lookup: output [B, D_offsets[T]] of out_dtype (F32 -> float32,
    F16 -> float16, BF16 -> uint16 holding bfloat16 bits)."""
    hsc, Do = _c(hash_size_cumsum, np.int64), _c(D_offsets, np.int32)
    wo = _c(weights_offsets, np.int64)
    idx, off = _c(indices, np.int64), _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    out = np.zeros((B, int(Do[T])), {F32: np.float32, F16: np.float16, BF16: np.uint16}[out_dtype])
    _check(_load().oracle_forward(T, B, _p(hsc), _p(Do), _p(wo), dtype_code(weights), _p(weights),
                                  _p(idx), _p(off), idx.size, _p(psw), int(bool(mean)), out_dtype,
                                  _p(out)))
    return out


def bucketize(T, B, row_bounds, indices, offsets, *, per_sample_weights=None, mean=False,
              cyclic=False):
    """A rank's batch split by the owner of each lookup's row (row_bounds [T, W+1];
    with cyclic, rank r owns rows r, r + W, ... and only row_bounds[:, W], the
    rows of every table, is read).

    Returns (send_offsets [W, T*B+1], send_indices, send_scales, send_counts [W]):
    owner r's lookups are send_indices[sum(send_counts[:r]) : ...], rows relative
    to r's range, scales = per-sample weight (1 if none) / L under mean pooling."""
    rb = _c(row_bounds, np.int64)
    W = rb.shape[1] - 1
    idx, off = _c(indices, np.int64), _c(offsets, np.int64)
    psw = _c(per_sample_weights, np.float32)
    so = np.zeros((W, T * B + 1), np.int64)
    si = np.zeros(idx.size, np.int64)
    ss = np.zeros(idx.size, np.float32)
    sc = np.zeros(W, np.int64)
    _check(_load().oracle_bucketize(T, B, W, _p(rb), int(bool(cyclic)), _p(idx), _p(off), idx.size, _p(psw),
                                    int(bool(mean)), _p(so), _p(si), _p(ss), _p(sc)))
    return so, si, ss, sc


def merge(T, B, W, recv_offsets, recv_indices, recv_scales):
    """The owner's batch after the exchange: CSR over T tables x W*B bags
    (bag s*B + b = source s's bag b), with its indices and scales."""
    ro = _c(recv_offsets, np.int64).reshape(W, T * B + 1)
    ri, rs = _c(recv_indices, np.int64), _c(recv_scales, np.float32)
    mo = np.zeros(T * W * B + 1, np.int64)
    mi = np.zeros(ri.size, np.int64)
    ms = np.zeros(ri.size, np.float32)
    _check(_load().oracle_merge(T, B, W, _p(ro), _p(ri), _p(rs), _p(mo), _p(mi), _p(ms)))
    return mo, mi, ms


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bf16_bits(x: float, r: int) -> int:
    return int(_load().oracle_sr_bf16(float(x), int(r)))


def sr_half_bits(x: float, r: int) -> int:
    return int(_load().oracle_sr_half(float(x), int(r)))


def double_to_half_bits(x: float) -> int:
    return int(_load().oracle_double_to_half(float(x)))


def half_bits_to_double(h: int) -> float:
    return float(_load().oracle_half_to_double(int(h)))


def double_to_bf16_bits(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def bf16_bits_to_double(h: int) -> float:
    return float(_load().oracle_bf16_to_double(int(h)))
