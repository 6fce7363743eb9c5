"""The row-sharded step with its exchange on two gloo ranks (CPU).

Every rank has its own batch and owns half the rows of every table. The same
orchestration the GPU ranks run (sparse_embedding_bag_gb300.shard: bucketize,
all-to-all of counts, offsets, indices and scales, merge, all-gather of
grad_output, backward on the rank's tables; forward with a reduce-scatter) is
driven here by the oracle in place of the library, over gloo. Rank 0 gathers
the shards and checks them against the unsharded oracle step on the global
batch (both ranks' bags side by side), and the forward against the unsharded
forward of each rank's own batch.
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


ROWS, DIMS, B = [97, 40, 300], [8, 16, 4], 24


def _batch(rank, weighted, optimizer):
    from sparse_embedding_bag_gb300 import synth
    rng = np.random.default_rng(100 + rank)
    # same model on both ranks (weights and state from seed 7), own lookups and gradients
    w = synth.make_bag_workload("sg", 7, ROWS, DIMS, B, rng.integers(0, 10, (3, B)),
                                lambda r, t, n: r.integers(0, ROWS[t], n).astype(np.int64),
                                optimizer=optimizer, weighted=weighted, momentum_init=0.5)
    own = synth.make_bag_workload("sg", 200 + rank, ROWS, DIMS, B, rng.integers(0, 10, (3, B)),
                                  lambda r, t, n: r.integers(0, ROWS[t], n).astype(np.int64),
                                  weighted=weighted)
    return w, own


class OracleOps:
    """The four library steps of one rank, computed by the oracle on CPU tensors."""

    def __init__(self, T, row_bounds, hsc, D_offsets, weights_offsets, cyclic):
        self.T, self.rb, self.cyclic = T, row_bounds, cyclic
        self.hsc, self.Do, self.wo = hsc, D_offsets, weights_offsets

    def bucketize(self, indices, offsets, N, B, psw, mode, send_offsets, send_indices, send_scales):
        import oracle
        so, si, ss, sc = oracle.bucketize(self.T, B, self.rb, indices[:N].numpy(), offsets.numpy(),
                                          per_sample_weights=None if psw is None else psw.numpy(),
                                          mean=(mode == 1), cyclic=self.cyclic)
        send_offsets.numpy()[:] = so
        send_indices.numpy()[:N] = si
        if send_scales is not None:
            send_scales.numpy()[:N] = ss
        return sc

    def merge(self, recv_offsets, recv_indices, recv_scales, n_recv, B, m_off, m_idx, m_scales):
        import oracle
        W = recv_offsets.shape[0]
        rs = np.ones(n_recv, np.float32) if recv_scales is None else recv_scales[:n_recv].numpy()
        mo, mi, ms = oracle.merge(self.T, B, W, recv_offsets.numpy(), recv_indices[:n_recv].numpy(), rs)
        m_off.numpy()[:] = mo
        m_idx.numpy()[:n_recv] = mi
        if m_scales is not None:
            m_scales.numpy()[:n_recv] = ms

    def backward(self, optimizer, weights, momentum, routed, grad, lr, eps):
        import oracle
        r = routed
        oracle.backward(self.T, r.B_all, self.hsc, self.Do, self.wo, weights.numpy(),
                        r.indices[:r.n].numpy(), r.offsets.numpy(), grad.numpy(),
                        optimizer=oracle.SGD if optimizer == "sgd" else oracle.ROWWISE_ADAGRAD,
                        lr=lr, eps=eps, momentum=None if momentum is None else momentum.numpy(),
                        per_sample_weights=None if r.scales is None else r.scales[:r.n].numpy())

    def forward(self, weights, routed, out, out_dtype):
        import oracle
        r = routed
        out.numpy()[:] = oracle.forward(self.T, r.B_all, self.hsc, self.Do, self.wo, weights.numpy(),
                                        r.indices[:r.n].numpy(), r.offsets.numpy(),
                                        per_sample_weights=None if r.scales is None else r.scales[:r.n].numpy())

    def close(self):
        pass


def _worker(rank, world, port, mode, out):
    import torch
    import torch.distributed as dist

    from sparse_embedding_bag_gb300 import shard as S
    from sparse_embedding_bag_gb300 import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        weighted, mean = "weighted" in mode, "mean" in mode
        optimizer = synth.ROWWISE_ADAGRAD if "adagrad" in mode else synth.SGD
        cyclic = "cyclic" in mode
        w, own = _batch(rank, weighted, optimizer)
        rb = S.even_row_bounds(ROWS, world)
        local, hsc, Do, wo = S.local_tables(ROWS, DIMS, rb, rank, world, cyclic)
        ops = OracleOps(len(ROWS), rb, hsc, Do, wo, cyclic)
        sb = S.RowShardedBags(ROWS, DIMS, rank, world, B, 4096, device="cpu", ops=ops, cyclic=cyclic)
        own_rows = S.owned_rows(ROWS, rb, rank, world, cyclic)
        weights = torch.from_numpy(np.concatenate(
            [w.weights[(w.weights_offsets[t] + own_rows[t][:, None] * DIMS[t] + np.arange(DIMS[t])).reshape(-1)]
             for t in range(len(ROWS))]).copy())
        mom = torch.from_numpy(np.concatenate(
            [w.momentum[w.hash_size_cumsum[t] + own_rows[t]] for t in range(len(ROWS))]).copy()) \
            if w.momentum is not None else None
        idx, off = torch.from_numpy(own.indices), torch.from_numpy(own.offsets)
        psw = None if own.per_sample_weights is None else torch.from_numpy(own.per_sample_weights)
        routed = sb.route(idx, off, own.N, B, psw, synth.MEAN if mean else synth.SUM)
        fwd = sb.forward(weights, routed).numpy()
        grad = torch.from_numpy(own.grad_output)
        if optimizer == synth.SGD:
            sb.backward_sgd(weights, routed, grad, w.lr)
        else:
            sb.backward_rowwise_adagrad(weights, mom, routed, grad, w.lr, w.eps)
        sb.close()
        shards = [None] * world
        dist.all_gather_object(shards, (weights.numpy(), None if mom is None else mom.numpy(), fwd,
                                        own.indices, own.offsets, own.per_sample_weights,
                                        own.grad_output))
        if rank == 0:
            out.put(_check(w, rb, shards, weighted, mean, optimizer, world, cyclic))
    finally:
        dist.destroy_process_group()


def _check(w, rb, shards, weighted, mean, optimizer, world, cyclic):
    import oracle
    from sparse_embedding_bag_gb300 import shard as S
    T = len(ROWS)
    # the unsharded forward of every rank's own batch
    for r in range(world):
        _, _, fwd, idx, off, psw, _ = shards[r]
        ref = oracle.forward(T, B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, w.weights,
                             idx, off, per_sample_weights=psw, mean=mean)
        if not np.allclose(fwd, ref, rtol=1e-5, atol=1e-6):
            return f"forward of rank {r} differs"
    # the unsharded step on the global batch: bag (t, s*B + b) = rank s's bag (t, b)
    gidx, goff, gpsw = [], [0], []
    for t in range(T):
        for s in range(world):
            _, _, _, idx, off, psw, _ = shards[s]
            for b in range(B):
                a, e = int(off[t * B + b]), int(off[t * B + b + 1])
                gidx.extend(idx[a:e].tolist())
                if psw is not None:
                    gpsw.extend(psw[a:e].tolist())
                goff.append(len(gidx))
    grad = np.concatenate([shards[s][6] for s in range(world)])
    ref_w = np.array(w.weights, copy=True)
    ref_m = None if w.momentum is None else w.momentum.copy()
    oracle.backward(T, world * B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, ref_w,
                    np.array(gidx, np.int64), np.array(goff, np.int64), grad,
                    optimizer=optimizer, lr=w.lr, eps=w.eps, momentum=ref_m,
                    per_sample_weights=np.array(gpsw, np.float32) if gpsw else None, mean=mean)
    for r in range(world):
        sw, sm = shards[r][0], shards[r][1]
        _, hsc, _, wo = S.local_tables(ROWS, DIMS, rb, r, world, cyclic)
        own_rows = S.owned_rows(ROWS, rb, r, world, cyclic)
        for t in range(T):
            D = DIMS[t]
            got = sw[wo[t]:wo[t] + own_rows[t].size * D]
            exp = ref_w[(w.weights_offsets[t] + own_rows[t][:, None] * D + np.arange(D)).reshape(-1)]
            exact = not (weighted or mean)
            if exact and not np.array_equal(got.view(np.uint32), exp.view(np.uint32)):
                return f"weights of rank {r} table {t} differ"
            if not exact and not np.allclose(got, exp, rtol=1e-6, atol=1e-7):
                return f"weights of rank {r} table {t} differ beyond rounding"
            if ref_m is not None:
                em = ref_m[w.hash_size_cumsum[t] + own_rows[t]]
                if not np.allclose(sm[hsc[t]:hsc[t + 1]], em, rtol=1e-6, atol=1e-9):
                    return f"state of rank {r} table {t} differs"
    if np.array_equal(ref_w, w.weights):
        return "nothing was updated"
    return "ok"


@pytest.mark.parametrize("mode", ["sum", "weighted_mean", "adagrad", "cyclic_sum",
                                  "cyclic_weighted_mean_adagrad"])
def test_row_sharded_step_two_gloo_ranks(mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert q.get(timeout=5) == "ok"
