"""The bench's row-sharded step (bench.py --op shard under torchrun) on two gloo
ranks on the CPU: the same function the GPU ranks run over NCCL, with the oracle
standing in for the library's four steps (bucketize, merge, forward, backward).
Rank 0 must print one JSON line of the bench contract that names the row
sharding and times the exchange, the forward and the backward separately."""
import io
import json
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _ops(w, rank, world):
    from test_shard_gloo import OracleOps
    from sparse_embedding_bag_gb300 import shard as S
    rb = S.even_row_bounds(w.rows, world)
    _, hsc, Do, wo = S.local_tables(w.rows, w.dims, rb, rank, world, cyclic=True)
    return OracleOps(w.T, rb, hsc, Do, wo, cyclic=True)


def _worker(rank, world, port, out):
    for p in (ROOT, HERE):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    buf = io.StringIO()
    stdout, sys.stdout = sys.stdout, buf
    try:
        bench.run_shard_dist(types.SimpleNamespace(steps=2, warmup=1, workload="tiny"), device="cpu",
                             ops_factory=_ops)
    finally:
        sys.stdout = stdout
        if dist.is_initialized():
            dist.destroy_process_group()
    if rank == 0:
        out.put(buf.getvalue())
    elif buf.getvalue().strip():
        out.put("rank 1 printed: " + buf.getvalue())


def test_sharded_bench_step_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    text = q.get(timeout=5)
    lines = [l for l in text.splitlines() if l.strip()]
    assert len(lines) == 1, text
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "stage_ms"):
        assert k in d, k
    assert d["n_gpus"] == 2 and d["steps"] == 2 and d["value"] > 0
    assert d["config"]["parallelism"] == "row-sharded, 2 ranks"
    assert set(d["stage_ms"]) == {"exchange", "forward", "backward"}
    assert q.empty()
