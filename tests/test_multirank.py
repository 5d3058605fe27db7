"""bench.py's multi-rank path on CPU (gloo, world size 2): each rank runs an
independent replica of the workload (its own seed, the same shapes, no data
exchanged) and the reported time is the slowest rank's; the reference arm runs
on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_replicas_gloo():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, os.path.join(HERE, "multirank_worker.py"), str(r), "2",
                               str(port)], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    # every rank sees the slowest rank's time
    assert outs[0]["slowest"] == outs[1]["slowest"] == 2.5
    # each rank draws its own replica: other seed, other data, same shapes
    assert outs[0]["seed"] != outs[1]["seed"]
    assert outs[0]["k_sum"] != outs[1]["k_sum"]
    assert outs[0]["offsets"] == outs[1]["offsets"]     # equal shards: same layout


def test_weak_scaling_value():
    import bench
    assert bench.weak_scaling_value(1000, 4, 2.0) == 1000 * 4 / 2e-3
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
                       "--workload", "c1_fp32_small"]) == 0
