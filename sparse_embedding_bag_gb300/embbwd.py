"""Thin ctypes binding of libembbwd (include/embbwd.h): same names, argument marshalling only.

Tensors are passed as raw device pointers (``tensor.data_ptr()``); host arrays
of the plan as numpy buffers. Every computation happens in the CUDA library;
there is no Python or CPU fallback: if the library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# EMBBWD_LIB selects another build of the library (e.g. for side-by-side timing).
LIB_PATH = os.environ.get("EMBBWD_LIB") or os.path.join(_PKG, "libembbwd.so")

EMB_OK, EMB_ERR_INVALID_ARG, EMB_ERR_UNSUPPORTED, EMB_ERR_INDEX_OUT_OF_RANGE = 0, 1, 2, 3
EMB_ERR_OOM, EMB_ERR_CUDA, EMB_ERR_TIMEOUT = 4, 5, 6
EMB_F32, EMB_F16, EMB_BF16 = 0, 1, 2
EMB_POOL_SUM, EMB_POOL_MEAN = 0, 1
EMB_NOBAG_AUTO, EMB_NOBAG_SORTED, EMB_NOBAG_ATOMIC = 0, 1, 2
EMB_FLAG_CHECK_INDICES = 0x1
EMB_FLAG_NO_PDL = 0x2
EMB_FLAG_STOCHASTIC_ROUNDING = 0x4
EMB_FLAG_NO_CLUSTER_FRONT = 0x8
EMB_FLAG_DEBUG_FORCE_TIMEOUT = 0x100

# Every symbol include/embbwd.h declares (checked by the tests against the header).
EXPORTS = ("emb_bwd_plan", "emb_plan_destroy", "emb_bag_bwd_sgd", "emb_bag_bwd_rowwise_adagrad",
           "emb_nobag_bwd_sgd", "emb_plan_status", "emb_plan_debug_runs", "emb_plan_set_profiling",
           "emb_plan_stage_ms", "emb_status_string", "emb_nobag_bwd_sgd_atomic_noalloc",
           "emb_bag_fwd", "emb_bag_bwd_adagrad", "emb_bag_bwd_dense_grad",
           "emb_nobag_bwd_dense_grad", "emb_plan_set_rounding", "emb_plan_get_rounding",
           "emb_shard_create", "emb_shard_create_cyclic", "emb_shard_destroy", "emb_shard_bucketize",
           "emb_shard_merge", "emb_shard_status")

_lock = threading.Lock()
_lib = None


class EmbError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def load(path: str = LIB_PATH):
    """Loads the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with sparse_embedding_bag_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64, u32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
        c_int = ctypes.c_int
        sig = {
            "emb_bwd_plan": [ctypes.POINTER(vp), c_int, i32, vp, vp, vp, vp, c_int, c_int, i64, i32, i32, u32],
            "emb_plan_destroy": [vp],
            "emb_bag_bwd_sgd": [vp, vp, vp, vp, i64, i32, vp, vp, c_int, f32, vp],
            "emb_bag_bwd_rowwise_adagrad": [vp, vp, vp, vp, vp, i64, i32, vp, vp, c_int, f32, f32, vp],
            "emb_nobag_bwd_sgd": [vp, vp, vp, vp, i64, i32, vp, f32, c_int, vp],
            "emb_plan_status": [vp],
            "emb_plan_debug_runs": [vp, i64, vp, vp, vp, vp, vp, vp],
            "emb_plan_set_profiling": [vp, c_int],
            "emb_plan_stage_ms": [vp, vp, i32],
            "emb_status_string": [c_int],
            "emb_nobag_bwd_sgd_atomic_noalloc": [c_int, i32, vp, vp, i32, vp, vp, vp, i64, i32, vp,
                                                 c_int, f32, vp, vp],
            "emb_bag_fwd": [vp, vp, vp, vp, i64, i32, vp, c_int, vp, c_int, vp],
            "emb_bag_bwd_adagrad": [vp, vp, vp, vp, vp, i64, i32, vp, vp, c_int, f32, f32, vp],
            "emb_bag_bwd_dense_grad": [vp, vp, vp, vp, i64, i32, vp, vp, c_int, vp],
            "emb_nobag_bwd_dense_grad": [vp, vp, vp, vp, i64, i32, vp, vp],
            "emb_plan_set_rounding": [vp, ctypes.c_uint64, ctypes.c_uint64],
            "emb_plan_get_rounding": [vp, vp, vp],
            "emb_shard_create": [ctypes.POINTER(vp), c_int, i32, i32, vp, i32],
            "emb_shard_create_cyclic": [ctypes.POINTER(vp), c_int, i32, i32, vp, i32],
            "emb_shard_destroy": [vp],
            "emb_shard_bucketize": [vp, vp, vp, i64, i32, vp, c_int, vp, vp, vp, vp, vp],
            "emb_shard_merge": [vp, vp, vp, vp, i64, i32, vp, vp, vp, vp],
            "emb_shard_status": [vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = c_int
        lib.emb_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().emb_status_string(int(status)).decode()


def _ptr(x):
    """Device pointer of a tensor, raw int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _host(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st, where):
    if st != EMB_OK:
        raise EmbError(st, where)
    return st


def emb_bwd_plan(device, T, hash_size_cumsum, D_offsets, weights_offsets, momentum_offsets,
                 weight_dtype, grad_dtype, max_N, max_B, max_segment_length_per_warp=0, flags=0):
    """Returns an opaque plan handle (int). Host arrays are copied by the library."""
    lib = load()
    hsc = _host(hash_size_cumsum, np.int64)
    Do = _host(D_offsets, np.int32)
    wo = _host(weights_offsets, np.int64)
    mo = _host(momentum_offsets, np.int64)
    out = ctypes.c_void_p()
    st = lib.emb_bwd_plan(ctypes.byref(out), int(device), int(T),
                          hsc.ctypes.data if hsc is not None else None,
                          Do.ctypes.data if Do is not None else None,
                          wo.ctypes.data if wo is not None else None,
                          mo.ctypes.data if mo is not None else None,
                          int(weight_dtype), int(grad_dtype), int(max_N), int(max_B),
                          int(max_segment_length_per_warp), int(flags))
    _check(st, "emb_bwd_plan")
    return out.value


def emb_plan_destroy(plan):
    return _check(load().emb_plan_destroy(plan), "emb_plan_destroy")


def emb_bag_bwd_sgd(plan, weights, indices, offsets, N, B, per_sample_weights, grad_output, mode,
                    lr, stream=None):
    st = load().emb_bag_bwd_sgd(plan, _ptr(weights), _ptr(indices), _ptr(offsets), int(N), int(B),
                                _ptr(per_sample_weights), _ptr(grad_output), int(mode),
                                float(lr), _stream(stream))
    return _check(st, "emb_bag_bwd_sgd")


def emb_bag_bwd_rowwise_adagrad(plan, weights, momentum, indices, offsets, N, B,
                                per_sample_weights, grad_output, mode, lr, eps, stream=None):
    st = load().emb_bag_bwd_rowwise_adagrad(plan, _ptr(weights), _ptr(momentum), _ptr(indices),
                                            _ptr(offsets), int(N), int(B),
                                            _ptr(per_sample_weights), _ptr(grad_output),
                                            int(mode), float(lr), float(eps), _stream(stream))
    return _check(st, "emb_bag_bwd_rowwise_adagrad")


def emb_nobag_bwd_sgd(plan, weights, indices, offsets, N, B, grad_output, lr,
                      path=EMB_NOBAG_AUTO, stream=None):
    st = load().emb_nobag_bwd_sgd(plan, _ptr(weights), _ptr(indices), _ptr(offsets), int(N),
                                  int(B), _ptr(grad_output), float(lr), int(path), _stream(stream))
    return _check(st, "emb_nobag_bwd_sgd")


def emb_bag_bwd_adagrad(plan, weights, momentum, indices, offsets, N, B, per_sample_weights,
                        grad_output, mode, lr, eps, stream=None):
    st = load().emb_bag_bwd_adagrad(plan, _ptr(weights), _ptr(momentum), _ptr(indices),
                                    _ptr(offsets), int(N), int(B), _ptr(per_sample_weights),
                                    _ptr(grad_output), int(mode), float(lr), float(eps),
                                    _stream(stream))
    return _check(st, "emb_bag_bwd_adagrad")


def emb_bag_bwd_dense_grad(plan, grad_weights, indices, offsets, N, B, per_sample_weights,
                           grad_output, mode, stream=None):
    st = load().emb_bag_bwd_dense_grad(plan, _ptr(grad_weights), _ptr(indices), _ptr(offsets),
                                       int(N), int(B), _ptr(per_sample_weights),
                                       _ptr(grad_output), int(mode), _stream(stream))
    return _check(st, "emb_bag_bwd_dense_grad")


def emb_nobag_bwd_dense_grad(plan, grad_weights, indices, offsets, N, B, grad_output, stream=None):
    st = load().emb_nobag_bwd_dense_grad(plan, _ptr(grad_weights), _ptr(indices), _ptr(offsets),
                                         int(N), int(B), _ptr(grad_output), _stream(stream))
    return _check(st, "emb_nobag_bwd_dense_grad")


def emb_bag_fwd(plan, weights, indices, offsets, N, B, per_sample_weights, mode, output,
                output_dtype, stream=None):
    st = load().emb_bag_fwd(plan, _ptr(weights), _ptr(indices), _ptr(offsets), int(N), int(B),
                            _ptr(per_sample_weights), int(mode), _ptr(output), int(output_dtype),
                            _stream(stream))
    return _check(st, "emb_bag_fwd")


def emb_plan_status(plan):
    """Returns the latched device status code (does not raise)."""
    return load().emb_plan_status(plan)


def emb_plan_debug_runs(plan, capacity):
    """Integer outputs of the last sorted call as numpy arrays."""
    cap = int(capacity)
    run_keys = np.zeros(max(cap, 1), np.int64)
    run_len = np.zeros(max(cap, 1), np.int32)
    cum = np.zeros(cap + 1, np.int32)
    long_ids = np.zeros(max(cap, 1), np.int32)
    nr = ctypes.c_int32(0)
    nl = ctypes.c_int32(0)
    st = load().emb_plan_debug_runs(plan, cap, run_keys.ctypes.data, run_len.ctypes.data,
                                    cum.ctypes.data, ctypes.addressof(nr), long_ids.ctypes.data,
                                    ctypes.addressof(nl))
    _check(st, "emb_plan_debug_runs")
    u, l = nr.value, nl.value
    return {"run_keys": run_keys[:u], "run_len": run_len[:u], "cum": cum[:u + 1],
            "num_runs": u, "long_ids": long_ids[:l]}


def emb_plan_set_profiling(plan, enable):
    return _check(load().emb_plan_set_profiling(plan, int(bool(enable))), "emb_plan_set_profiling")


def emb_plan_set_rounding(plan, seed, next_call=0):
    return _check(load().emb_plan_set_rounding(plan, int(seed) & (2 ** 64 - 1),
                                               int(next_call) & (2 ** 64 - 1)),
                  "emb_plan_set_rounding")


def emb_plan_get_rounding(plan):
    """(seed, next call number) of the plan's stochastic rounding."""
    out = np.zeros(2, np.uint64)
    _check(load().emb_plan_get_rounding(plan, out.ctypes.data, out.ctypes.data + 8),
           "emb_plan_get_rounding")
    return int(out[0]), int(out[1])


def emb_plan_stage_ms(plan, n=5):
    out = np.zeros(n, np.float32)
    _check(load().emb_plan_stage_ms(plan, out.ctypes.data, n), "emb_plan_stage_ms")
    return out


def emb_nobag_bwd_sgd_atomic_noalloc(device, T, hash_size_cumsum, weights_offsets, D, weights,
                                     indices, offsets, N, B, grad_output, grad_dtype, lr,
                                     device_status=None, stream=None):
    """Allocation-free unpooled atomic SGD; table arrays are device tensors (int64)."""
    st = load().emb_nobag_bwd_sgd_atomic_noalloc(int(device), int(T), _ptr(hash_size_cumsum),
                                                 _ptr(weights_offsets), int(D), _ptr(weights),
                                                 _ptr(indices), _ptr(offsets), int(N), int(B),
                                                 _ptr(grad_output), int(grad_dtype), float(lr),
                                                 _ptr(device_status), _stream(stream))
    return _check(st, "emb_nobag_bwd_sgd_atomic_noalloc")


# ---- row-wise sharding (exchange step)

def emb_shard_create(device, T, W, row_bounds, max_B):
    """Shard map of one rank; row_bounds host int64 [T, W+1]. Returns a handle (int)."""
    rb = _host(row_bounds, np.int64)
    assert rb.size == T * (W + 1)
    out = ctypes.c_void_p()
    _check(load().emb_shard_create(ctypes.byref(out), int(device), int(T), int(W), rb.ctypes.data,
                                   int(max_B)), "emb_shard_create")
    return out.value


def emb_shard_create_cyclic(device, T, W, rows, max_B):
    """Cyclic shard map (rank r owns rows r, r + W, ...); rows host int64 [T]."""
    rw = _host(rows, np.int64)
    assert rw.size == T
    out = ctypes.c_void_p()
    _check(load().emb_shard_create_cyclic(ctypes.byref(out), int(device), int(T), int(W),
                                          rw.ctypes.data, int(max_B)), "emb_shard_create_cyclic")
    return out.value


def emb_shard_destroy(shard):
    return _check(load().emb_shard_destroy(shard), "emb_shard_destroy")


def emb_shard_bucketize(shard, indices, offsets, N, B, per_sample_weights, mode, send_offsets,
                        send_indices, send_scales, stream=None):
    """Splits the batch by row owner into the send buffers (send_offsets a device
    int64 tensor [W, T*B+1]); returns the per-owner lookup counts (host int64 [W]).
    Synchronises the stream."""
    counts = np.zeros(int(send_offsets.shape[0]), np.int64)
    st = load().emb_shard_bucketize(shard, _ptr(indices), _ptr(offsets), int(N), int(B),
                                    _ptr(per_sample_weights), int(mode), _ptr(send_offsets),
                                    _ptr(send_indices), _ptr(send_scales), counts.ctypes.data,
                                    _stream(stream))
    _check(st, "emb_shard_bucketize")
    return counts


def emb_shard_merge(shard, recv_offsets, recv_indices, recv_scales, n_recv, B, merged_offsets,
                    merged_indices, merged_scales, stream=None):
    st = load().emb_shard_merge(shard, _ptr(recv_offsets), _ptr(recv_indices), _ptr(recv_scales),
                                int(n_recv), int(B), _ptr(merged_offsets), _ptr(merged_indices),
                                _ptr(merged_scales), _stream(stream))
    return _check(st, "emb_shard_merge")


def emb_shard_status(shard):
    return load().emb_shard_status(shard)
