"""Parity at the full size of the large skewed workload (64 tables x 2M rows,
D=128 fp16 weights + fp32 row-wise state, B=65536, ~1.25e8 lookups, Zipf(1.2)
ids with hot rows hit hundreds of thousands of times), in the launch
configuration the bench times. The whole step runs on the GPU through the C ABI;
the oracle, which cannot hold this step, recomputes sampled rows one by one
(the hottest rows, random touched rows, random untouched rows) from every lookup
of each: fp16 weights within 1 ulp, state within rtol 1e-4 / atol 1e-5,
untouched rows bit-identical."""
import pytest

from _full_size import sampled_rows_check
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


def test_large_skewed_full_size_sampled_rows():
    import torch
    w = synth.large_on_device(0, device="cuda")
    dw = dev.to_device(w, "cuda")
    assert dw.weights.data_ptr() == w.weights.data_ptr()  # updated in place, seen through w
    plan = dev.make_plan(w)
    try:
        def step():
            dev.step(plan, dw)
            assert E.emb_plan_status(plan) == E.EMB_OK
        checked = sampled_rows_check(w, step)
    finally:
        E.emb_plan_destroy(plan)
        del dw, w
        torch.cuda.empty_cache()
    assert checked >= 50
