"""Host side of the sequence-parallel exchange of packed NVFP4 KV head shards.

The segment size comes from the C library (no GPU needed); the exchange is one
all-to-all of equal segments through torch.distributed, run here as two gloo
ranks on the CPU.  Each rank packs its own quantized tensor (the layout of
tests/exchange_layout.py), exchanges, and checks that it received shard r of
rank r's tensor for every r, in rank order.
"""
import os
import socket
import subprocess
import sys

import numpy as np

from exchange_layout import pad16, seg_bytes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_segment_bytes_follow_the_layout():
    import nvfp4_block_quantization_gb300 as nv

    nv.load_library()
    for (T, H, D, P) in [(7040, 24, 128, 2), (7040, 24, 128, 4), (880, 24, 128, 3), (16, 4, 16, 4), (1, 2, 64, 1)]:
        for wm in (False, True):
            assert nv.kv_shard_bytes(T, H, D, P, wm) == seg_bytes(T, H, D, P, wm)
            assert nv.kv_shard_bytes(T, H, D, P, wm) % 16 == 0
    assert nv.kv_shard_bytes(7040, 24, 128, 5, True) == 0     # 24 heads do not split in 5
    assert nv.kv_shard_bytes(7040, 24, 120, 2, True) == 0     # D % 16 != 0
    # the bytes each rank sends per tensor and per layer, against bf16: 3.5x fewer
    T, H, D, P = 7040, 24, 128, 2
    sent = (P - 1) * seg_bytes(T, H, D, P, True)
    bf16 = (P - 1) * T * (H // P) * D * 2
    assert 3.5 < bf16 / sent < 3.6


WORKER = r"""
import os, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
import numpy as np, torch, torch.distributed as dist
import nvfp4_block_quantization_gb300 as nv
from exchange_layout import pack, unpack
dist.init_process_group("gloo")
rank, P = dist.get_rank(), dist.get_world_size()
T, H, D = 24, 6, 32
def tensor(r):
    rng = np.random.default_rng(100 + r)
    return (rng.integers(0, 256, (T, H, D // 2), dtype=np.uint8), rng.integers(0, 127, (T, H, D // 16), dtype=np.uint8),
            np.float32(0.01 * (r + 1)), rng.standard_normal((H, D)).astype(np.float32))
codes, scales, g, mean = tensor(rank)
segs = torch.from_numpy(pack(codes, scales, g, mean, P))
got = nv.kv_exchange_head_shards(segs).numpy()
c, s, gs, ms = unpack(got, T, H, D, P, True)
hs = H // P
for r in range(P):
    rc, rsc, rg, rm = tensor(r)
    assert np.array_equal(c[r * T:(r + 1) * T], rc[:, rank * hs:(rank + 1) * hs])
    assert np.array_equal(s[r * T:(r + 1) * T], rsc[:, rank * hs:(rank + 1) * hs])
    assert gs[r] == rg
    assert np.array_equal(ms[r], rm[rank * hs:(rank + 1) * hs])
dist.barrier()
dist.destroy_process_group()
print("ok", rank)
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_exchange_head_shards():
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
        assert p.returncode == 0, err[-3000:]
        outs.append(out.strip())
    assert sorted(outs) == ["ok 0", "ok 1"]
