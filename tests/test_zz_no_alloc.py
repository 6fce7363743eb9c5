"""The allocation-free entry point, emb_nobag_bwd_sgd_atomic_noalloc.

It serves callers that cannot allocate device memory when they run the update
(inside a CUDA graph capture, under a runtime that owns all device memory, or
where the library must not call the device allocator): no plan, scratch in a
fixed static device array. This file is collected last so that a run stopping
at its first failure has already run every other test.

Checked through the C ABI against the existing entry point (a plan plus
emb_nobag_bwd_sgd with the atomic path) and against the CPU oracle's unpooled
SGD step, within the parity tolerance, on two calls in a row each, so that the
shared scratch being left over from the previous call is exercised. Malformed
device-side table arrays (a misaligned or negative weights offset, a
hash_size_cumsum that does not increase) must be reported in device_status with
nothing updated, and the next valid call must start clean.
"""
import numpy as np
import pytest

from _helpers import oracle_step
from sparse_embedding_bag_gb300 import device as dev
from sparse_embedding_bag_gb300 import embbwd as E
from sparse_embedding_bag_gb300 import synth

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_embedding_bag_gb300 import build
    build.build()
    E.load()


def _workload(seed, grad_dtype=synth.F32):
    rng = np.random.default_rng(seed)
    rows, D, B = [700, 3000, 45], 64, 16
    return synth.make_bag_workload(
        "noalloc", seed, rows, [D] * 3, B, rng.integers(0, 60, (3, B)),
        lambda r, t, n: synth.sample_zipf(r, rows[t], 1.1, n), nobag=True, grad_dtype=grad_dtype)


@pytest.mark.parametrize("grad_dtype", [synth.F32, synth.F16, synth.BF16])
def test_noalloc_matches_planned_atomic_path_twice(grad_dtype):
    import torch
    w = _workload(11, grad_dtype)
    ref = dev.to_device(w)
    new = dev.to_device(w)
    hsc = torch.from_numpy(w.hash_size_cumsum).cuda()
    wo = torch.from_numpy(w.weights_offsets).cuda()
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    plan = dev.make_plan(w)
    try:
        for _ in range(2):
            E.emb_nobag_bwd_sgd(plan, ref.weights, ref.indices, ref.offsets, w.N, w.B,
                                ref.grad_output, w.lr, E.EMB_NOBAG_ATOMIC)
            E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, hsc, wo, int(w.dims[0]), new.weights,
                                               new.indices, new.offsets, w.N, w.B,
                                               new.grad_output, w.grad_dtype, w.lr, status)
            torch.cuda.synchronize()
            assert E.emb_plan_status(plan) == E.EMB_OK
            assert int(status.item()) == 0
            np.testing.assert_allclose(new.weights.cpu().numpy(), ref.weights.cpu().numpy(),
                                       rtol=RTOL, atol=ATOL)
    finally:
        E.emb_plan_destroy(plan)
    assert not np.array_equal(new.weights.cpu().numpy(), w.weights)  # it did update


@pytest.mark.parametrize("grad_dtype", [synth.F32, synth.F16])
def test_noalloc_matches_oracle(grad_dtype):
    import torch
    w = _workload(13, grad_dtype)
    d = dev.to_device(w)
    hsc = torch.from_numpy(w.hash_size_cumsum).cuda()
    wo = torch.from_numpy(w.weights_offsets).cuda()
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, hsc, wo, int(w.dims[0]), d.weights, d.indices,
                                       d.offsets, w.N, w.B, d.grad_output, w.grad_dtype, w.lr, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    exp, _ = oracle_step(w)
    np.testing.assert_allclose(d.weights.cpu().numpy(), exp, rtol=RTOL, atol=ATOL)


def test_noalloc_reports_errors_and_limits():
    import torch
    w = _workload(12)
    d = dev.to_device(w)
    hsc = torch.from_numpy(w.hash_size_cumsum).cuda()
    wo = torch.from_numpy(w.weights_offsets).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = int(w.dims[0])
    # beyond the stated maximum number of lookups: rejected on the host
    with pytest.raises(E.EmbError) as e:
        E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, hsc, wo, D, d.weights, d.indices, d.offsets,
                                           (1 << 22) + 1, w.B, d.grad_output, w.grad_dtype, w.lr,
                                           status)
    assert e.value.status == E.EMB_ERR_INVALID_ARG
    # an index outside its table: reported in device_status, nothing updated
    bad = d.indices.clone()
    bad[w.N // 2] = 10**9
    before = d.weights.clone()
    E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, hsc, wo, D, d.weights, bad, d.offsets, w.N, w.B,
                                       d.grad_output, w.grad_dtype, w.lr, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    assert torch.equal(d.weights, before)
    # the next valid call starts clean
    E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, hsc, wo, D, d.weights, d.indices, d.offsets, w.N,
                                       w.B, d.grad_output, w.grad_dtype, w.lr, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert not torch.equal(d.weights, before)


@pytest.mark.parametrize("case", ["misaligned_offset", "negative_offset", "flat_cumsum"])
def test_noalloc_rejects_malformed_tables_on_device(case):
    """The device-side table arrays are checked before the scatter runs: a bad one
    sets bit 2 of device_status and leaves the weights untouched; the next valid
    call succeeds."""
    import torch
    w = _workload(14)
    d = dev.to_device(w)
    hsc_h, wo_h = w.hash_size_cumsum.copy(), w.weights_offsets.copy()
    if case == "misaligned_offset":
        wo_h[1] += 2
    elif case == "negative_offset":
        wo_h[2] = -4
    else:
        hsc_h[2] = hsc_h[1]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = int(w.dims[0])
    before = d.weights.clone()
    E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, torch.from_numpy(hsc_h).cuda(), torch.from_numpy(wo_h).cuda(),
                                       D, d.weights, d.indices, d.offsets, w.N, w.B, d.grad_output,
                                       w.grad_dtype, w.lr, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    assert torch.equal(d.weights, before)
    E.emb_nobag_bwd_sgd_atomic_noalloc(0, w.T, torch.from_numpy(w.hash_size_cumsum).cuda(),
                                       torch.from_numpy(w.weights_offsets).cuda(), D, d.weights,
                                       d.indices, d.offsets, w.N, w.B, d.grad_output, w.grad_dtype,
                                       w.lr, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert not torch.equal(d.weights, before)
