"""Seeded synthetic inputs for the embedding backward workloads.

This module only draws random arrays and lays them out in the CSR / flat-table
form the library consumes. It holds none of the backward pass's arithmetic, so
both the CPU oracle (in tests) and the CUDA path can take their inputs from it.

Workloads (all seeded with numpy ``default_rng`` sub-streams; the large skewed
one is drawn on the device with a seeded ``torch.Generator``):

* ``tiny``: 2 tables (1000, 500 rows), D=16 fp32, B=64, bag length U{0..4}
  (empty bags occur), uniform ids, sum pooling, SGD.
* ``dlrm``: 8 tables x 100k rows, D=64 fp32, B=2048, bag length U{1..20},
  bounded Zipf(1.05) ids, sum pooling, row-wise Adagrad.
* ``mixed``: 26 tables, rows log-uniform in [1e3, 1e6], D drawn per table
  from {32, 64, 128, 256}, fp16 weights, fp32 grad, B=16384, bag length
  Poisson(15), per-sample weights U(0,1), mean pooling, row-wise Adagrad,
  bounded Zipf(1.05) ids.
* ``lm``: one 128256 x 4096 fp32 table, bf16 grad [32768, 4096], bounded
  Zipf(1.1) token ids, unpooled, SGD.
* ``large``: 64 tables x 2M rows, D=128 fp16 weights, fp32 momentum and grad,
  B=65536, bag length power law on [1, 500] with mean 30, bounded Zipf(1.2)
  ids, sum pooling, row-wise Adagrad.

Bounded Zipf(a) on E rows: P(rank k) proportional to k^-a for k = 1..E, drawn
by inverse CDF; rank k maps to row k-1, so the hot rows of a table are its
first rows.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32, F16, BF16 = 0, 1, 2
SGD, ROWWISE_ADAGRAD = 0, 1
SUM, MEAN = 0, 1


@dataclasses.dataclass
class Workload:
    """One backward step's inputs, host (numpy) or device (torch) arrays."""
    name: str
    T: int
    B: int
    rows: np.ndarray                 # int64[T]
    dims: np.ndarray                 # int32[T]
    hash_size_cumsum: np.ndarray     # int64[T+1]
    D_offsets: np.ndarray            # int32[T+1]
    weights_offsets: np.ndarray      # int64[T]
    momentum_offsets: Optional[np.ndarray]  # int64[T] or None (= hash_size_cumsum[:T])
    weight_dtype: int
    grad_dtype: int
    optimizer: int
    pooling: int
    nobag: bool
    lr: float                        # exact fp32 value
    eps: float                       # exact fp32 value
    indices: object                  # int64[N]
    offsets: object                  # int64[B*T+1]
    grad_output: object              # [B, sum D] (bag) or [N, D] (nobag); bf16 held as uint16 bits
    weights: object                  # flat, weight storage dtype (bf16 as uint16 bits)
    momentum: object = None          # float32[sum rows] or None
    per_sample_weights: object = None  # float32[N] or None

    @property
    def N(self) -> int:
        return int(self.indices.shape[0])

    @property
    def max_D(self) -> int:
        return int(np.max(self.dims))


def _f32(x: float) -> float:
    return float(np.float32(x))


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def zipf_cdf(E: int, a: float) -> np.ndarray:
    k = np.arange(1, E + 1, dtype=np.float64)
    c = np.cumsum(k ** (-a))
    return c / c[-1]


def sample_zipf(rng, E: int, a: float, n: int, cdf=None) -> np.ndarray:
    """Bounded Zipf(a) ranks on 1..E by inverse CDF, returned as rows 0..E-1."""
    if cdf is None:
        cdf = zipf_cdf(E, a)
    u = rng.random(n)
    r = np.searchsorted(cdf, u, side="right")
    return np.minimum(r, E - 1).astype(np.int64)


def power_law_exponent_for_mean(mean: float, kmax: int) -> float:
    """Exponent a with E[k] = mean for P(k) proportional to k^-a on 1..kmax (bisection)."""
    k = np.arange(1, kmax + 1, dtype=np.float64)

    def m(a):
        p = k ** (-a)
        return float((k * p).sum() / p.sum())

    lo, hi = 0.0, 4.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if m(mid) > mean:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _to_storage(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return x.astype(np.float32)
    if dtype == F16:
        return x.astype(np.float16)
    import torch
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def table_layout(rows, dims):
    rows = np.asarray(rows, np.int64)
    dims = np.asarray(dims, np.int32)
    T = rows.size
    hsc = np.zeros(T + 1, np.int64)
    hsc[1:] = np.cumsum(rows)
    Do = np.zeros(T + 1, np.int32)
    Do[1:] = np.cumsum(dims)
    wo = np.zeros(T, np.int64)
    wo[1:] = np.cumsum(rows * dims.astype(np.int64))[:-1]
    return hsc, Do, wo


def make_bag_workload(name, seed, rows, dims, B, lengths, id_sampler, *, weight_dtype=F32,
                      grad_dtype=F32, optimizer=SGD, pooling=SUM, weighted=False, lr=0.01,
                      eps=1e-8, momentum_init=0.0, nobag=False):
    """Generic pooled (or unpooled) workload.

    lengths: int64[T, B] bag lengths. id_sampler(rng, t, n) -> int64[n] rows of table t.
    For nobag the grad is [N, D] (uniform D) and the CSR only assigns lookups to tables.
    """
    r_ids, r_w, r_g, r_psw, r_m = _streams(seed, 5)
    rows = np.asarray(rows, np.int64)
    dims = np.asarray(dims, np.int32)
    T = rows.size
    hsc, Do, wo = table_layout(rows, dims)
    lengths = np.asarray(lengths, np.int64).reshape(T, B)
    offsets = np.zeros(T * B + 1, np.int64)
    offsets[1:] = np.cumsum(lengths.reshape(-1))
    N = int(offsets[-1])
    indices = np.empty(N, np.int64)
    for t in range(T):
        a, b = int(offsets[t * B]), int(offsets[(t + 1) * B])
        indices[a:b] = id_sampler(r_ids, t, b - a)
    total_w = int((rows * dims.astype(np.int64)).sum())
    weights = _to_storage(r_w.uniform(-0.1, 0.1, total_w).astype(np.float32), weight_dtype)
    if nobag:
        assert np.all(dims == dims[0])
        g = r_g.standard_normal((N, int(dims[0])), dtype=np.float32)
    else:
        g = r_g.standard_normal((B, int(Do[-1])), dtype=np.float32)
    grad = _to_storage(g, grad_dtype)
    psw = r_psw.random(N, dtype=np.float32) if weighted else None
    momentum = None
    if optimizer == ROWWISE_ADAGRAD:
        if momentum_init:
            momentum = r_m.uniform(0.0, momentum_init, int(hsc[-1])).astype(np.float32)
        else:
            momentum = np.zeros(int(hsc[-1]), np.float32)
    return Workload(name=name, T=T, B=B, rows=rows, dims=dims, hash_size_cumsum=hsc,
                    D_offsets=Do, weights_offsets=wo, momentum_offsets=None,
                    weight_dtype=weight_dtype, grad_dtype=grad_dtype, optimizer=optimizer,
                    pooling=pooling, nobag=nobag, lr=_f32(lr), eps=_f32(eps), indices=indices,
                    offsets=offsets, grad_output=grad, weights=weights, momentum=momentum,
                    per_sample_weights=psw)


def tiny(seed: int = 0) -> Workload:
    rng = _streams(seed, 6)[5]
    rows, dims, B = [1000, 500], [16, 16], 64
    lengths = rng.integers(0, 5, size=(2, B))
    return make_bag_workload("tiny", seed, rows, dims, B, lengths,
                             lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                             optimizer=SGD, lr=0.01)


def dlrm(seed: int = 0) -> Workload:
    rng = _streams(seed, 6)[5]
    T, E, D, B = 8, 100_000, 64, 2048
    lengths = rng.integers(1, 21, size=(T, B))
    cdf = zipf_cdf(E, 1.05)
    return make_bag_workload("dlrm", seed, [E] * T, [D] * T, B, lengths,
                             lambda r, t, n: sample_zipf(r, E, 1.05, n, cdf),
                             optimizer=ROWWISE_ADAGRAD, lr=0.01, eps=1e-8)


def mixed(seed: int = 0, B: int = 16384, zipf_a: Optional[float] = 1.05) -> Workload:
    """zipf_a=None draws uniform ids (the alternate case)."""
    rng = _streams(seed, 6)[5]
    T = 26
    rows = np.round(10 ** rng.uniform(3.0, 6.0, T)).astype(np.int64)
    dims = rng.choice(np.array([32, 64, 128, 256], np.int32), T)
    lengths = rng.poisson(15, size=(T, B))
    cdfs = {}

    def ids(r, t, n):
        if zipf_a is None:
            return r.integers(0, rows[t], n).astype(np.int64)
        if t not in cdfs:
            cdfs[t] = zipf_cdf(int(rows[t]), zipf_a)
        return sample_zipf(r, int(rows[t]), zipf_a, n, cdfs[t])

    return make_bag_workload("mixed", seed, rows, dims, B, lengths, ids, weight_dtype=F16,
                             optimizer=ROWWISE_ADAGRAD, pooling=MEAN, weighted=True, lr=0.01,
                             eps=1e-8)


def lm(seed: int = 0, tokens: int = 8 * 4096, vocab: int = 128256, D: int = 4096) -> Workload:
    cdf = zipf_cdf(vocab, 1.1)
    lengths = np.array([[tokens]], np.int64)
    return make_bag_workload("lm", seed, [vocab], [D], 1, lengths,
                             lambda r, t, n: sample_zipf(r, vocab, 1.1, n, cdf),
                             grad_dtype=BF16, optimizer=SGD, lr=1e-3, nobag=True)


LARGE = dict(T=64, E=2_000_000, D=128, B=65536, kmax=500, mean_len=30.0, zipf_a=1.2)


def large_on_device(seed: int = 0, device="cuda", T=None, B=None, E=None, tables=None):
    """The large skewed workload, drawn on the device (too big for host-side numpy).

    Returns a Workload whose arrays are torch tensors on `device`. Bag lengths
    follow P(k) ~ k^-a on 1..500 with a chosen so the mean is 30; ids are
    bounded Zipf(1.2) per table (rank k -> row k-1).

    Every table draws from its own generator (seeded seed * 2^16 + t): its bag
    lengths, its ids, its weights and its [B, D] column block of grad_output.
    `tables` = k draws only the first k tables, which are then exactly the
    first k tables of the full workload (tables are independent, so that cut is
    a workload of its own with the same per-table statistics).
    """
    import torch
    p = dict(LARGE)
    T = p["T"] if T is None else T
    B = p["B"] if B is None else B
    E = p["E"] if E is None else E
    D = p["D"]
    T_draw = T if tables is None else min(int(tables), T)
    gens = []
    for t in range(T_draw):
        g = torch.Generator(device=device)
        g.manual_seed(seed * 65536 + t)
        gens.append(g)
    a_len = power_law_exponent_for_mean(p["mean_len"], p["kmax"])
    k = torch.arange(1, p["kmax"] + 1, dtype=torch.float64, device=device)
    len_cdf = torch.cumsum(k ** (-a_len), 0)
    len_cdf /= len_cdf[-1].clone()
    lengths = torch.empty(T_draw * B, dtype=torch.int64, device=device)
    for t in range(T_draw):
        u = torch.rand(B, generator=gens[t], device=device, dtype=torch.float64)
        lengths[t * B:(t + 1) * B] = torch.searchsorted(len_cdf, u, right=True).clamp_(max=p["kmax"] - 1) + 1
    offsets = torch.zeros(T_draw * B + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(lengths, 0)
    N = int(offsets[-1].item())
    kk = torch.arange(1, E + 1, dtype=torch.float64, device=device)
    id_cdf = torch.cumsum(kk ** (-p["zipf_a"]), 0)
    id_cdf /= id_cdf[-1].clone()
    indices = torch.empty(N, dtype=torch.int64, device=device)
    bounds = offsets[::B].cpu().numpy()
    for t in range(T_draw):
        a, b = int(bounds[t]), int(bounds[t + 1])
        uu = torch.rand(b - a, generator=gens[t], device=device, dtype=torch.float64)
        indices[a:b] = torch.searchsorted(id_cdf, uu, right=True).clamp_(max=E - 1)
    rows = np.full(T_draw, E, np.int64)
    dims = np.full(T_draw, D, np.int32)
    hsc, Do, wo = table_layout(rows, dims)
    weights = torch.empty(T_draw * E * D, dtype=torch.float16, device=device)
    for t in range(T_draw):
        s = t * E * D
        weights[s:s + E * D] = (torch.rand(E * D, generator=gens[t], device=device) * 0.2 - 0.1).to(torch.float16)
    momentum = torch.zeros(T_draw * E, dtype=torch.float32, device=device)
    grad = torch.empty(B, T_draw * D, device=device, dtype=torch.float32)
    for t in range(T_draw):
        grad[:, t * D:(t + 1) * D] = torch.randn(B, D, generator=gens[t], device=device, dtype=torch.float32)
    T = T_draw
    return Workload(name="large", T=T, B=B, rows=rows, dims=dims, hash_size_cumsum=hsc,
                    D_offsets=Do, weights_offsets=wo, momentum_offsets=None, weight_dtype=F16,
                    grad_dtype=F32, optimizer=ROWWISE_ADAGRAD, pooling=SUM, nobag=False,
                    lr=_f32(0.01), eps=_f32(1e-8), indices=indices, offsets=offsets,
                    grad_output=grad, weights=weights, momentum=momentum,
                    per_sample_weights=None)


BY_NAME = {"tiny": tiny, "dlrm": dlrm, "mixed": mixed, "lm": lm}
