"""bench.py's multi-rank host logic on CPU: two ranks over gloo.

The GEMM path itself has no exchange step (replicas only: every rank runs
the whole product on its own GPU), so what N > 1 adds is host logic -- the
barrier around the timed region, the maximum of the step time over ranks,
the whole-job rate (all ranks' work / the slowest rank's time), and the rule
that only rank 0 prints.  These tests run that logic as real processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.init("gloo")
rank = d.rank
# rank r "took" 10 + 5 r ms for 2e12 FLOP; rank 1 arrives late at the barrier
if rank == 1:
    time.sleep(0.3)
t0 = time.time()
d.barrier()
waited = time.time() - t0
ms, rate = bench.job_rate(d, 2e12, 10.0 + 5.0 * rank)
print(json.dumps({{"rank": rank, "world": d.world, "ms": ms, "rate": rate, "waited": waited}}))
d.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ)
    env.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    return env


def test_two_ranks_share_the_slowest_time():
    port = _free_port()
    code = CHILD.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    for o in outs:
        assert o["world"] == 2
        assert o["ms"] == 15.0                     # the slower rank's time, on both ranks
        # 2 ranks x 2e12 FLOP in 15 ms
        assert abs(o["rate"] - 2 * 2e12 / 15e-3 / 1e12) < 1e-9
    assert outs[0]["waited"] > 0.1                 # rank 0 waited for rank 1 at the barrier


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    if d.world != 1:
        pytest.skip("running under a launcher")
    ms, rate = bench.job_rate(d, 1e12, 4.0)
    assert ms == 4.0 and abs(rate - 250.0) < 1e-9


def test_reference_arm_on_other_ranks_exits_quietly():
    """Under torchrun only rank 0 runs the reference (CPU oracle) arm; the
    other ranks exit 0 at once, without output and without joining a group."""
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
