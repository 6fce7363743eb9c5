"""Moves a seeded workload to the GPU and calls the matching C-ABI entry point.

Marshalling only: tensors are allocated with PyTorch and handed to libembbwd as
raw pointers; the backward pass itself runs in the library's CUDA kernels.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import embbwd as E
from .synth import BF16, ROWWISE_ADAGRAD, SGD, Workload


@dataclasses.dataclass
class DeviceWorkload:
    w: Workload
    indices: object
    offsets: object
    grad_output: object
    weights: object
    momentum: object
    per_sample_weights: object


def _t(x, device):
    import torch
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.to(device).contiguous()
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        a = a.view(np.int16)  # bf16 bits: only the pointer matters to the library
    return torch.from_numpy(a).to(device)


def to_device(w: Workload, device="cuda") -> DeviceWorkload:
    return DeviceWorkload(w=w, indices=_t(w.indices, device), offsets=_t(w.offsets, device),
                          grad_output=_t(w.grad_output, device), weights=_t(w.weights, device),
                          momentum=_t(w.momentum, device),
                          per_sample_weights=_t(w.per_sample_weights, device))


def make_plan(w: Workload, device_index: int = 0, max_N=None, max_B=None,
              max_segment_length_per_warp: int = 0, flags: int = 0):
    return E.emb_bwd_plan(device_index, w.T, w.hash_size_cumsum, w.D_offsets, w.weights_offsets,
                          w.momentum_offsets, w.weight_dtype, w.grad_dtype,
                          w.N if max_N is None else max_N, w.B if max_B is None else max_B,
                          max_segment_length_per_warp, flags)


def step(plan, dw: DeviceWorkload, path: int = E.EMB_NOBAG_AUTO, stream=None, N=None):
    """One backward + update through the C ABI (asynchronous on `stream`)."""
    w = dw.w
    n = w.N if N is None else N
    if w.nobag:
        return E.emb_nobag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, n, w.B,
                                   dw.grad_output, w.lr, path, stream)
    if w.optimizer == SGD:
        return E.emb_bag_bwd_sgd(plan, dw.weights, dw.indices, dw.offsets, n, w.B,
                                 dw.per_sample_weights, dw.grad_output, w.pooling, w.lr, stream)
    assert w.optimizer == ROWWISE_ADAGRAD
    return E.emb_bag_bwd_rowwise_adagrad(plan, dw.weights, dw.momentum, dw.indices, dw.offsets, n,
                                         w.B, dw.per_sample_weights, dw.grad_output, w.pooling,
                                         w.lr, w.eps, stream)


def forward(plan, dw: DeviceWorkload, out_dtype: int = 0, out=None, stream=None):
    """Forward pooled lookup through the C ABI into `out` (allocated if None):
    a [B, sum D] tensor of out_dtype (0 fp32, 1 fp16, 2 bf16). Returns `out`."""
    import torch
    w = dw.w
    if out is None:
        tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[out_dtype]
        out = torch.empty((w.B, int(w.D_offsets[-1])), dtype=tdt, device=dw.weights.device)
    E.emb_bag_fwd(plan, dw.weights, dw.indices, dw.offsets, w.N, w.B, dw.per_sample_weights,
                  w.pooling, out, out_dtype, stream)
    return out


def weights_numpy(dw: DeviceWorkload) -> np.ndarray:
    """Device weights back as numpy in the workload's storage representation."""
    a = dw.weights.cpu().numpy()
    if dw.w.weight_dtype == BF16:
        a = a.view(np.uint16)
    return a
