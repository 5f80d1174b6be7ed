"""The bench's multi-process path on CPU: two gloo ranks on 127.0.0.1 (one process each, as torchrun
launches them) agree on the world size, reduce the step time to the maximum over ranks, and draw
different shards of the global batch."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_the_max_and_shard_the_batch():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "tests", "_dist_worker.py")], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    assert [o["rank"] for o in outs] == [0, 1]
    assert all(o["world"] == 2 for o in outs)
    assert all(o["max_ms"] == 3.0 for o in outs)          # max of 1.5 and 3.0, seen by both ranks
    assert outs[0]["seed"] != outs[1]["seed"]
