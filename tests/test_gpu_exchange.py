"""Head-shard pack/unpack kernels of the sequence-parallel exchange, on the GPU.

P ranks are emulated on one GPU by P quantized tensors; the all-to-all itself
(torch.distributed) is exercised on the CPU in test_exchange_host.py.  Packing
must reproduce the documented segment layout byte for byte; unpacking the
segments a rank receives must give back, for every source rank, exactly its
shard of codes, scales, tensor scale and mean, and the cache read over the
unpacked P groups must equal the read of each source tensor's shard.
"""
import numpy as np
import pytest

from exchange_layout import pack, unpack

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    from nvfp4_block_quantization_gb300.build import build

    build()
    import nvfp4_block_quantization_gb300 as nv

    nv.load_library()
    return nv


@pytest.mark.parametrize("P,smooth", [(2, True), (3, True), (3, False), (6, True)])
def test_pack_exchange_unpack_round_trip(nv, P, smooth):
    from nvfp4_block_quantization_gb300 import workloads as W

    T, H, D = 40, 6, 64
    ranks = []
    for r in range(P):
        x = W.to_bf16_bits(W.random_kv(300 + r, T, H, D))
        q = nv.kv_smooth_quant(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda(), smooth)
        seg = nv.kv_shard_bytes(T, H, D, P, smooth)
        out = torch.zeros((P, seg), dtype=torch.uint8, device="cuda")
        nv.kv_pack_head_shards(q, P, out=out)
        torch.cuda.synchronize()
        host = dict(codes=q.codes.cpu().numpy(), scales=q.scales.cpu().numpy(), g=float(q.tensor_scale.item()),
                    mean=None if q.mean is None else q.mean.cpu().numpy())
        ref = pack(host["codes"], host["scales"], host["g"], host["mean"], P)
        assert np.array_equal(out.cpu().numpy(), ref)
        ranks.append((q, out, host))
    hs = H // P
    for me in range(P):
        # what rank `me` receives from an all-to-all: segment `me` of every rank, in rank order
        recv = torch.stack([ranks[r][1][me] for r in range(P)])
        codes, scales, gs, means = nv.kv_unpack_head_shards(recv, T, H, D, P, smooth)
        torch.cuda.synchronize()
        rc, rs, rg, rm = unpack(recv.cpu().numpy(), T, H, D, P, smooth)
        assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
        assert np.array_equal(gs.cpu().numpy(), rg)
        if smooth:
            assert np.array_equal(means.cpu().numpy(), rm)
        for r in range(P):
            h = ranks[r][2]
            assert np.array_equal(rc[r * T:(r + 1) * T], h["codes"][:, me * hs:(me + 1) * hs])
            assert np.array_equal(rs[r * T:(r + 1) * T], h["scales"][:, me * hs:(me + 1) * hs])
        # the cache read over the P received groups equals each source's own read of the shard
        got = nv.kv_dequant(codes, scales, gs, mean=means.reshape(P, -1) if smooth else None, tokens_per_group=T)
        for r in range(P):
            q = ranks[r][0]
            full = nv.kv_dequant(q.codes, q.scales, q.tensor_scale, mean=q.mean)
            a = got[r * T:(r + 1) * T].view(torch.int16).cpu().numpy()
            b = full[:, me * hs:(me + 1) * hs].contiguous().view(torch.int16).cpu().numpy()
            assert np.array_equal(a, b)
