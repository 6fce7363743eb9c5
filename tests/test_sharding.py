"""Row-sharded backward on two gloo ranks (CPU) equals the unsharded one.

Each rank owns a contiguous row range of every table (the vocabulary sharding
of "Function _embedding_bwd_kernel": lookups outside the rank's range add
nothing there). Every rank runs the oracle on its shard, the shards are
gathered over gloo, and rank 0 checks them bit for bit against the unsharded
oracle step. The GPU path itself is single-GPU; this pins the sharding
semantics a multi-GPU deployment relies on.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _workload(weighted):
    from sparse_embedding_bag_gb300 import synth
    rng = np.random.default_rng(5)
    rows, dims, B = [97, 40, 300], [8, 16, 4], 50
    return synth.make_bag_workload("shard", 5, rows, dims, B, rng.integers(0, 12, (3, B)),
                                   lambda r, t, n: r.integers(0, rows[t], n).astype(np.int64),
                                   optimizer=synth.ROWWISE_ADAGRAD, weighted=weighted)


def _shard(w, rank, world):
    """The rank's local problem: its row range of every table, lookups outside dropped."""
    lo = [w.rows[t] * rank // world for t in range(w.T)]
    hi = [w.rows[t] * (rank + 1) // world for t in range(w.T)]
    idx, off, psw = [], [0], []
    for bt in range(w.T * w.B):
        t = bt // w.B
        for i in range(int(w.offsets[bt]), int(w.offsets[bt + 1])):
            if lo[t] <= w.indices[i] < hi[t]:
                idx.append(int(w.indices[i]) - lo[t])
                if w.per_sample_weights is not None:
                    psw.append(w.per_sample_weights[i])
        off.append(len(idx))
    local_rows = np.array([hi[t] - lo[t] for t in range(w.T)], np.int64)
    hsc = np.concatenate([[0], np.cumsum(local_rows)]).astype(np.int64)
    wo = np.concatenate([[0], np.cumsum(local_rows * w.dims)[:-1]]).astype(np.int64)
    weights = np.concatenate([w.weights[w.weights_offsets[t] + lo[t] * w.dims[t]:
                                        w.weights_offsets[t] + hi[t] * w.dims[t]] for t in range(w.T)])
    mom = np.concatenate([w.momentum[w.hash_size_cumsum[t] + lo[t]:w.hash_size_cumsum[t] + hi[t]]
                          for t in range(w.T)])
    return (hsc, wo, weights.copy(), mom.copy(), np.array(idx, np.int64), np.array(off, np.int64),
            None if w.per_sample_weights is None else np.array(psw, np.float32))


def _worker(rank, world, port, weighted, out):
    import torch
    import torch.distributed as dist

    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _workload(weighted)
        hsc, wo, weights, mom, idx, off, psw = _shard(w, rank, world)
        if idx.size:
            oracle.backward(w.T, w.B, hsc, w.D_offsets, wo, weights, idx, off, w.grad_output,
                            optimizer=w.optimizer, lr=w.lr, eps=w.eps, momentum=mom,
                            per_sample_weights=psw)
        shards = [None] * world
        dist.all_gather_object(shards, (weights, mom))
        if rank == 0:
            ref_w = w.weights.copy()
            ref_m = w.momentum.copy()
            oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, ref_w,
                            w.indices, w.offsets, w.grad_output, optimizer=w.optimizer, lr=w.lr,
                            eps=w.eps, momentum=ref_m, per_sample_weights=w.per_sample_weights)
            # reassemble table by table from the shards
            got_w = np.empty_like(ref_w)
            got_m = np.empty_like(ref_m)
            for t in range(w.T):
                pos_w, pos_m = w.weights_offsets[t], w.hash_size_cumsum[t]
                for r in range(world):
                    lo = w.rows[t] * r // world
                    hi = w.rows[t] * (r + 1) // world
                    s_hsc = np.concatenate([[0], np.cumsum([w.rows[u] * (r + 1) // world - w.rows[u] * r // world
                                                            for u in range(w.T)])])
                    s_wo = np.concatenate([[0], np.cumsum([(w.rows[u] * (r + 1) // world - w.rows[u] * r // world) * w.dims[u]
                                                           for u in range(w.T)])])
                    sw, sm = shards[r]
                    n = (hi - lo) * w.dims[t]
                    got_w[pos_w:pos_w + n] = sw[s_wo[t]:s_wo[t] + n]
                    got_m[pos_m:pos_m + hi - lo] = sm[s_hsc[t]:s_hsc[t] + hi - lo]
                    pos_w += n
                    pos_m += hi - lo
            ok = (np.array_equal(got_w.view(np.uint32), ref_w.view(np.uint32)) and
                  np.array_equal(got_m.view(np.uint32), ref_m.view(np.uint32)))
            out.put(ok)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("weighted", [False, True])
def test_row_sharded_equals_unsharded(oracle_mod, weighted):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, weighted, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
