"""Row-wise sharded embedding bags over a process group (one rank per GPU).

Every rank trains on its own batch and owns a contiguous row range of every
table, the vocabulary sharding of "Function _embedding_bwd_kernel" (tinygrad:
a device owns one slice of the rows, lookups outside it add nothing there), or
with cyclic=True the rows congruent to its rank modulo W (row k*W + r is local
row k of rank r), which spreads a skewed id distribution over all ranks.
One step on every rank:

  route     the library buckets the rank's lookups by row owner
            (emb_shard_bucketize), an all-to-all delivers every owner its
            lookups from all ranks, and the library lays them out as one batch
            of W*B bags per table (emb_shard_merge);
  backward  an all-gather of grad_output gives the W*B gradient rows in rank
            order, then the ordinary backward of the library runs on the
            rank's own tables with B' = W*B (per-lookup scales as weights);
  forward   the library's pooled lookup with B' = W*B gives this rank's partial
            sums of every rank's bags; a reduce-scatter returns each rank its own.

The collectives go through torch.distributed (NCCL on GPUs); every lookup,
scale and update is computed by the library. The `ops` argument exists so that
the same orchestration can be driven by other implementations of the four
library steps (the CPU tests drive it with the oracle over gloo).
"""
from __future__ import annotations

import numpy as np

from . import embbwd as E


def even_row_bounds(rows, world):
    """Row ranges of W ranks, as even as possible: int64 [T, W+1]."""
    rows = np.asarray(rows, np.int64)
    return np.array([[int(r) * k // world for k in range(world + 1)] for r in rows], np.int64)


def owned_rows(rows, row_bounds, rank, world, cyclic=False):
    """Global rows of every table that the rank owns, in its local order."""
    if cyclic:
        return [np.arange(rank, int(r), world, dtype=np.int64) for r in rows]
    rb = np.asarray(row_bounds, np.int64)
    return [np.arange(rb[t, rank], rb[t, rank + 1], dtype=np.int64) for t in range(len(rows))]


def local_tables(rows, dims, row_bounds, rank, world=None, cyclic=False):
    """The rank's own tables: (rows, hash_size_cumsum, D_offsets, weights_offsets)
    of its rows of every table, weights packed table after table."""
    if cyclic:
        local = np.array([(int(r) - rank + world - 1) // world for r in rows], np.int64)
    else:
        rb = np.asarray(row_bounds, np.int64)
        local = (rb[:, rank + 1] - rb[:, rank]).astype(np.int64)
    dims = np.asarray(dims, np.int64)
    hsc = np.concatenate([[0], np.cumsum(local)]).astype(np.int64)
    D_offsets = np.concatenate([[0], np.cumsum(dims)]).astype(np.int32)
    weights_offsets = np.concatenate([[0], np.cumsum(local * dims)[:-1]]).astype(np.int64)
    return local, hsc, D_offsets, weights_offsets


class CudaOps:
    """The four library steps of one rank (C ABI calls on its device)."""

    def __init__(self, device, T, world, row_bounds, max_B, plan, rows=None, cyclic=False):
        if cyclic:
            self.shard = E.emb_shard_create_cyclic(device, T, world, rows, max_B)
        else:
            self.shard = E.emb_shard_create(device, T, world, row_bounds, max_B)
        self.plan = plan

    def bucketize(self, indices, offsets, N, B, psw, mode, send_offsets, send_indices, send_scales):
        return E.emb_shard_bucketize(self.shard, indices, offsets, N, B, psw, mode, send_offsets,
                                     send_indices, send_scales)

    def merge(self, recv_offsets, recv_indices, recv_scales, n_recv, B, m_off, m_idx, m_scales):
        E.emb_shard_merge(self.shard, recv_offsets, recv_indices, recv_scales, n_recv, B, m_off,
                          m_idx, m_scales)
        st = E.emb_shard_status(self.shard)
        if st != E.EMB_OK:
            raise E.EmbError(st, "emb_shard_merge")

    def backward(self, optimizer, weights, momentum, routed, grad, lr, eps):
        r = routed
        if optimizer == "sgd":
            E.emb_bag_bwd_sgd(self.plan, weights, r.indices, r.offsets, r.n, r.B_all, r.scales, grad,
                              E.EMB_POOL_SUM, lr)
        else:
            E.emb_bag_bwd_rowwise_adagrad(self.plan, weights, momentum, r.indices, r.offsets, r.n,
                                          r.B_all, r.scales, grad, E.EMB_POOL_SUM, lr, eps)
        st = E.emb_plan_status(self.plan)
        if st != E.EMB_OK:
            raise E.EmbError(st, "sharded backward")

    def forward(self, weights, routed, out, out_dtype):
        r = routed
        E.emb_bag_fwd(self.plan, weights, r.indices, r.offsets, r.n, r.B_all, r.scales,
                      E.EMB_POOL_SUM, out, out_dtype)

    def close(self):
        E.emb_shard_destroy(self.shard)


class Routed:
    """One rank's lookups after the exchange: a batch of B_all = W*B bags per table."""

    def __init__(self, offsets, indices, scales, n, B, B_all):
        self.offsets, self.indices, self.scales = offsets, indices, scales
        self.n, self.B, self.B_all = n, B, B_all


class RowShardedBags:
    """One rank's part of row-wise sharded embedding bags.

    rows, dims: the full tables; row_bounds [T, W+1] (default: even ranges), or
    cyclic=True for the modulo-W map;
    max_B: the largest per-rank batch; max_N: the most lookups one rank sends or
    receives per step. The rank's weights and state are its local tables
    (local_tables()); all ranks pass the same B, pooling and weighting.
    """

    def __init__(self, rows, dims, rank, world, max_B, max_N, *, row_bounds=None, cyclic=False,
                 group=None, device="cuda", weight_dtype=0, grad_dtype=0, flags=0, ops=None):
        import torch
        self.rows, self.dims = np.asarray(rows, np.int64), np.asarray(dims, np.int64)
        self.T, self.rank, self.world = len(self.rows), rank, world
        self.cyclic = cyclic
        self.row_bounds = even_row_bounds(rows, world) if row_bounds is None else np.asarray(row_bounds, np.int64)
        self.max_B, self.max_N, self.group = max_B, max_N, group
        self.device = torch.device(device)
        self.local_rows, self.hsc, self.D_offsets, self.weights_offsets = local_tables(
            self.rows, self.dims, self.row_bounds, rank, world, cyclic)
        self.plan = None
        if ops is None:
            dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
            self.plan = E.emb_bwd_plan(dev_index, self.T, self.hsc, self.D_offsets,
                                       self.weights_offsets, None, weight_dtype, grad_dtype,
                                       max_N, world * max_B, 0, flags)
            ops = CudaOps(dev_index, self.T, world, self.row_bounds, max_B, self.plan, self.rows, cyclic)
        self.ops = ops
        BT = self.T * max_B
        i64 = torch.int64
        self.send_offsets = torch.empty((world, BT + 1), dtype=i64, device=self.device)
        self.send_indices = torch.empty(max(max_N, 1), dtype=i64, device=self.device)
        self.send_scales = torch.empty(max(max_N, 1), dtype=torch.float32, device=self.device)

    # -- collectives (torch.distributed)
    def _a2a(self, out, inp, out_splits=None, in_splits=None):
        import torch.distributed as dist
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)

    def route(self, indices, offsets, N, B, per_sample_weights=None, mode=E.EMB_POOL_SUM):
        """Delivers every rank the lookups of its rows from all ranks' batches."""
        import torch
        assert B <= self.max_B and N <= self.max_N
        W, BT = self.world, self.T * B
        need_scales = per_sample_weights is not None or mode == E.EMB_POOL_MEAN
        send_off = self.send_offsets.view(-1)[:W * (BT + 1)].view(W, BT + 1)
        send_sc = self.send_scales if need_scales else None
        counts = self.ops.bucketize(indices, offsets, N, B, per_sample_weights, mode, send_off,
                                    self.send_indices, send_sc)
        send_counts = torch.as_tensor(np.asarray(counts, np.int64), device=self.device)
        recv_counts = torch.empty_like(send_counts)
        self._a2a(recv_counts, send_counts)
        rc = recv_counts.cpu().numpy().astype(np.int64)
        sc = np.asarray(counts, np.int64)
        n_recv = int(rc.sum())
        if n_recv > self.max_N:
            raise ValueError(f"rank {self.rank} receives {n_recv} lookups, above max_N={self.max_N}")
        recv_off = torch.empty(W * (BT + 1), dtype=torch.int64, device=self.device)
        self._a2a(recv_off, send_off.reshape(-1).contiguous())
        recv_idx = torch.empty(max(n_recv, 1), dtype=torch.int64, device=self.device)
        self._a2a(recv_idx[:n_recv], self.send_indices[:N], rc.tolist(), sc.tolist())
        recv_sc = None
        if need_scales:
            recv_sc = torch.empty(max(n_recv, 1), dtype=torch.float32, device=self.device)
            self._a2a(recv_sc[:n_recv], self.send_scales[:N], rc.tolist(), sc.tolist())
        m_off = torch.empty(W * BT + 1, dtype=torch.int64, device=self.device)
        m_idx = torch.empty(max(n_recv, 1), dtype=torch.int64, device=self.device)
        m_sc = torch.empty(max(n_recv, 1), dtype=torch.float32, device=self.device) if need_scales else None
        self.ops.merge(recv_off.view(W, BT + 1), recv_idx, recv_sc, n_recv, B, m_off, m_idx, m_sc)
        return Routed(m_off, m_idx, m_sc, n_recv, B, W * B)

    def gather_grad(self, grad_output):
        """[B, sum D] per rank -> [W*B, sum D] in rank order."""
        import torch
        import torch.distributed as dist
        g = grad_output.contiguous()
        out = torch.empty((self.world * g.shape[0],) + tuple(g.shape[1:]), dtype=g.dtype, device=g.device)
        dist.all_gather_into_tensor(out, g, group=self.group)
        return out

    def backward_sgd(self, weights, routed, grad_output, lr):
        if routed.n:
            self.ops.backward("sgd", weights, None, routed, self.gather_grad(grad_output), lr, 0.0)
        else:
            self.gather_grad(grad_output)  # every rank takes part in the collective

    def backward_rowwise_adagrad(self, weights, momentum, routed, grad_output, lr, eps):
        if routed.n:
            self.ops.backward("rowwise_adagrad", weights, momentum, routed,
                              self.gather_grad(grad_output), lr, eps)
        else:
            self.gather_grad(grad_output)

    def forward(self, weights, routed):
        """Pooled fp32 output of this rank's own B bags, [B, sum D]: the owners'
        fp32 partial sums added by the reduce-scatter."""
        import torch
        import torch.distributed as dist
        sumD = int(self.dims.sum())
        partial = torch.zeros((routed.B_all, sumD), dtype=torch.float32, device=self.device)
        if routed.n:
            self.ops.forward(weights, routed, partial, 0)
        out = torch.empty((routed.B, sumD), dtype=torch.float32, device=self.device)
        dist.reduce_scatter_tensor(out, partial, group=self.group)
        return out

    def close(self):
        self.ops.close()
        if self.plan is not None:
            E.emb_plan_destroy(self.plan)
            self.plan = None
