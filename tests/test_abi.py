"""CPU-side checks of the C ABI: the library builds, loads, exports every symbol
include/embbwd.h declares, and rejects malformed arguments on the host before
any CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from sparse_embedding_bag_gb300 import build as B
from sparse_embedding_bag_gb300 import embbwd as E

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "embbwd.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return E.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(emb_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    decl = declared_functions()
    assert len(decl) >= 10
    assert sorted(E.EXPORTS) == decl
    for name in decl:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert E.status_string(code) not in ("", "unknown status")
    assert E.status_string(99) == "unknown status"


def _plan(lib, T=2, hsc=(0, 10, 30), Do=(0, 8, 16), wo=(0, 80), mo=None, wdt=0, gdt=0,
          max_N=100, max_B=4, thr=0, flags=0, out=True):
    p = ctypes.c_void_p()
    arr = lambda a, t: None if a is None else np.ascontiguousarray(a, t)
    h, d, w, m = arr(hsc, np.int64), arr(Do, np.int32), arr(wo, np.int64), arr(mo, np.int64)
    keep = (h, d, w, m)
    st = lib.emb_bwd_plan(ctypes.byref(p) if out else None, 0, T,
                          *(None if a is None else a.ctypes.data for a in keep),
                          wdt, gdt, max_N, max_B, thr, flags)
    return st, p


@pytest.mark.parametrize("kw", [
    dict(T=0),
    dict(T=5000),
    dict(hsc=(0, 10, 10)),            # empty / shared table
    dict(hsc=(1, 10, 30)),            # must start at 0
    dict(Do=(0, 6, 12)),              # D not a multiple of 4
    dict(Do=(0, 8, 8)),               # D = 0
    dict(Do=(0, 8, 8 + 8192)),        # D above the supported maximum
    dict(wo=(0, 82)),                 # row starts must stay 16-byte aligned
    dict(max_N=1 << 30),
    dict(max_N=-1),
    dict(max_B=0),
    dict(wdt=3),
    dict(gdt=-1),
    dict(hsc=(0, 1 << 31, 1 << 33)),  # more than 2^32 rows
    dict(out=False),
])
def test_plan_rejects_bad_arguments_without_cuda(lib, kw):
    st, p = _plan(lib, **kw)
    assert st == E.EMB_ERR_INVALID_ARG
    assert not p.value


def test_calls_reject_null_plan(lib):
    assert lib.emb_bag_bwd_sgd(None, None, None, None, 0, 1, None, None, 0, 0.1, None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_bag_bwd_rowwise_adagrad(None, None, None, None, None, 0, 1, None, None, 0, 0.1,
                                           0.0, None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_nobag_bwd_sgd(None, None, None, None, 0, 1, None, 0.1, 0, None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_status(None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_debug_runs(None, 0, None, None, None, None, None, None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_set_profiling(None, 1) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_stage_ms(None, None, 0) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_destroy(None) == E.EMB_OK


def test_header_declares_status_codes_used_by_binding():
    text = open(HEADER).read()
    for name in ("EMB_OK = 0", "EMB_ERR_INVALID_ARG = 1", "EMB_ERR_UNSUPPORTED = 2",
                 "EMB_ERR_INDEX_OUT_OF_RANGE = 3", "EMB_ERR_OOM = 4", "EMB_ERR_CUDA = 5",
                 "EMB_ERR_TIMEOUT = 6", "EMB_F32 = 0", "EMB_F16 = 1", "EMB_BF16 = 2",
                 "EMB_POOL_SUM = 0", "EMB_POOL_MEAN = 1", "EMB_NOBAG_ATOMIC = 2"):
        assert name in text
    assert "EMB_FLAG_DEBUG_FORCE_TIMEOUT 0x100u" in text
    assert E.EMB_FLAG_DEBUG_FORCE_TIMEOUT == 0x100
    # every plan flag of the header, with the binding's value
    import re
    flags = dict(re.findall(r"#define (EMB_FLAG_\w+) (0x[0-9a-fA-F]+)u", text))
    assert set(flags) == {"EMB_FLAG_CHECK_INDICES", "EMB_FLAG_NO_PDL", "EMB_FLAG_STOCHASTIC_ROUNDING",
                          "EMB_FLAG_NO_CLUSTER_FRONT", "EMB_FLAG_DEBUG_FORCE_TIMEOUT"}
    for name, value in flags.items():
        assert getattr(E, name) == int(value, 16), name
    assert len(set(flags.values())) == len(flags)  # distinct bits


def _shard(lib, T=2, W=2, rb=((0, 5, 10), (0, 3, 7)), max_B=4, out=True, cyclic=False):
    p = ctypes.c_void_p()
    if cyclic:
        a = np.ascontiguousarray(rb, np.int64)
        st = lib.emb_shard_create_cyclic(ctypes.byref(p) if out else None, 0, T, W, a.ctypes.data, max_B)
    else:
        a = np.ascontiguousarray(rb, np.int64)
        st = lib.emb_shard_create(ctypes.byref(p) if out else None, 0, T, W, a.ctypes.data, max_B)
    return st, p


@pytest.mark.parametrize("kw", [
    dict(T=0),
    dict(W=0),
    dict(W=300, rb=[[0] * 300 + [10], [0] * 300 + [7]]),   # more than 256 ranks
    dict(rb=((1, 5, 10), (0, 3, 7))),                        # ranges must start at row 0
    dict(rb=((0, 6, 5), (0, 3, 7))),                         # decreasing bounds
    dict(rb=((0, 0, 0), (0, 3, 7))),                         # a table without rows
    dict(max_B=0),
    dict(max_B=1 << 29),                                     # W * T * max_B >= 2^31
    dict(out=False),
    dict(cyclic=True, rb=(10, 0)),                           # cyclic: a table without rows
])
def test_shard_create_rejects_bad_arguments_without_cuda(lib, kw):
    st, p = _shard(lib, **kw)
    assert st == E.EMB_ERR_INVALID_ARG
    assert not p.value


def test_shard_and_rounding_calls_reject_null_handles(lib):
    assert lib.emb_shard_bucketize(None, None, None, 0, 1, None, 0, None, None, None, None, None) == \
        E.EMB_ERR_INVALID_ARG
    assert lib.emb_shard_merge(None, None, None, None, 0, 1, None, None, None, None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_shard_status(None) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_shard_destroy(None) == E.EMB_OK
    assert lib.emb_plan_set_rounding(None, 1, 2) == E.EMB_ERR_INVALID_ARG
    assert lib.emb_plan_get_rounding(None, None, None) == E.EMB_ERR_INVALID_ARG
