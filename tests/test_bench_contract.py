"""The bench's reference arm on the CPU: one JSON line with the keys of the
bench contract (the GPU arm needs a device and runs in the GPU suite's bench
step), and nothing from ranks other than 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = _run({})
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "lookups/s" and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_are_silent():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_launches_per_step_follow_the_front():
    # the kernels a step launches, which the bench line reports as gpu_launches
    sys.path.insert(0, ROOT)
    import bench
    # multi-block front: histogram, the passes, run-length, reduce
    launches, names, per_step = bench.step_stages(False, False, 2)
    assert per_step == 5 and sum(launches) == 5 and names[1] == "radix_sort"
    # the small-batch front: one launch for the whole front, then the reduce
    launches, names, per_step = bench.step_stages(False, True, 2)
    assert per_step == 2 and launches == [1, 0, 0, 0, 1] and names[0] == "cluster_front"
    # unpooled atomic scatter: the index check and the scatter
    assert bench.step_stages(True, False, 3)[2] == 2
    # row-wise Adagrad on rows of several 1024-wide chunks: the reduce twice
    assert bench.step_stages(False, False, 3, reduce_launches=2)[2] == 7
    assert bench.step_stages(False, True, 3, reduce_launches=2)[2] == 3
