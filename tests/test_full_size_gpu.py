"""Parity at the full size of the large skewed workload (64 tables x 2M rows,
D=128 fp16 weights + fp32 row-wise state, B=65536, ~1.25e8 lookups, Zipf(1.2)
ids with hot rows hit hundreds of thousands of times), in the launch
configuration the bench times. The whole step runs on the GPU through the C ABI.

* Integer outputs (sorted unique linear indices, run lengths, run starts, long
  runs as a set) bit-exact on the first two tables: their keys are the smallest,
  so the first runs of the full sort are exactly the runs of those two tables,
  which the oracle computes whole (~4e6 lookups).
* Floating point: the oracle, which cannot hold this step, recomputes sampled
  rows one by one (the hottest rows, random touched rows, random untouched rows)
  from every lookup of each: fp16 weights within 1 ulp, state within rtol 1e-4 /
  atol 1e-5, untouched rows bit-identical."""
import numpy as np
import pytest

import oracle
from _full_size import sampled_rows_check
from _helpers import compare_runs
from sparse_embedding_bag_gb300 import device as dev
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def large():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_embedding_bag_gb300 import build
    build.build()
    E.load()
    w = synth.large_on_device(0, device="cuda")
    dw = dev.to_device(w, "cuda")
    assert dw.weights.data_ptr() == w.weights.data_ptr()  # updated in place, seen through w
    plan = dev.make_plan(w)
    yield w, dw, plan
    E.emb_plan_destroy(plan)
    del dw, w
    torch.cuda.empty_cache()


def test_large_skewed_full_size_sampled_rows(large):
    w, dw, plan = large

    def step():
        dev.step(plan, dw)
        assert E.emb_plan_status(plan) == E.EMB_OK
    assert sampled_rows_check(w, step) >= 50


def test_large_skewed_full_size_integer_outputs_first_two_tables(large):
    w, dw, plan = large
    dev.step(plan, dw)
    assert E.emb_plan_status(plan) == E.EMB_OK
    got = E.emb_plan_debug_runs(plan, w.N)
    B, T2 = w.B, 2
    off = w.offsets[:T2 * B + 1].cpu().numpy()
    idx = w.indices[:int(off[-1])].cpu().numpy()
    exp = oracle.runs(T2, B, w.hash_size_cumsum[:T2 + 1], idx, off, 32)
    U2 = exp["num_runs"]
    assert got["num_runs"] > U2 and got["run_keys"][U2] >= w.hash_size_cumsum[T2]
    lids = got["long_ids"]
    part = {"num_runs": U2, "run_keys": got["run_keys"][:U2], "run_len": got["run_len"][:U2],
            "cum": got["cum"][:U2 + 1], "long_ids": np.sort(lids[lids < U2])}
    compare_runs(part, exp)
