"""Multi-rank host logic of bench.py: two gloo ranks on the CPU.

The path does not shard (each rank is an independent replica of the step), so the only
cross-rank code is the set-up, the barrier around the timed region and the max over
ranks of the measured time; these run here as world_size-2 gloo processes.
"""
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys
sys.path.insert(0, sys.argv[1])
import bench
ws, rank, local = bench.dist_setup()
assert (ws, rank, local) == (2, int(os.environ["RANK"]), int(os.environ["LOCAL_RANK"]))
bench.barrier(ws)
t = bench.max_over_ranks(ws, 10.0 + rank)  # rank-dependent "times"
assert t == 11.0, t
bench.barrier(ws)
import torch.distributed as dist
dist.destroy_process_group()
print("ok", rank)
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_barrier_and_max_time():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(r), LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out.strip())
    assert sorted(outs) == ["ok 0", "ok 1"]
