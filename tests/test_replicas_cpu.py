"""Multi-replica bench logic on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job rate (units of all ranks / that time)."""
import json
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_take_the_slowest_rank():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "replica_worker.py")], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["ws"] == 2 and o["local"] == o["rank"]
        assert o["ms_max"] == 15.0                       # the slower rank's window
        assert abs(o["rate"] - 100 * 2 / 15e-3) < 1e-6    # both ranks' units over it


def test_single_process_needs_no_group():
    sys.path.insert(0, os.path.dirname(HERE))
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_rate(10, 1, 5.0) == 2000.0
