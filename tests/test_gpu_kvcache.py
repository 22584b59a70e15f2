"""GPU: the multi-shot NVFP4 KV cache through the C ABI.

Chunks of K and V are quantized straight into the pool slots the manager hands out
(LongLive-2.0 summary page, inference step 7), and each chunk's view (step 9: global
sink, shot sink, rolling window) is expanded by the gathered read.  Bars:
  * the gathered read is bit-exact against the oracle's dequant of the same pool
    bytes, each frame with its own slot's tensor scale (and mean, for K);
  * every view frame's pool rows hold exactly the codes, scales, tensor scale and
    mean that a standalone call gives for the chunk the frame belongs to, so no
    live frame was overwritten by a later chunk.
"""
import numpy as np
import pytest

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


def dev(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def host(t):
    return t.detach().cpu().numpy()


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def same_bits_nan(a, b):
    """bf16 bit patterns equal, any NaN matching any NaN."""
    fa = (a.astype(np.uint32) << 16).view(np.float32)
    fb = (b.astype(np.uint32) << 16).view(np.float32)
    both_nan = np.isnan(fa) & np.isnan(fb)
    return bool(np.all((a == b) | both_nan))


def check_view(nv, oracle, cache, pk, pv, ref, L):
    fi, fr, fs = cache.view()
    F = cache.state.frames_per_chunk
    ck, sk, gk, mk = host(pk.codes), host(pk.scales), host(pk.g), host(pk.mean)
    cv, sv, gv = host(pv.codes), host(pv.scales), host(pv.g)
    # the pool holds each view frame's chunk as a standalone call quantizes it
    for f, r, s in zip(fi, fr, fs):
        k = int(f) // F
        a = (int(f) % F) * L
        rk, rv = ref[k]
        assert np.array_equal(ck[r:r + L], rk["codes"][a:a + L]) and np.array_equal(sk[r:r + L], rk["scales"][a:a + L])
        assert np.array_equal(cv[r:r + L], rv["codes"][a:a + L]) and np.array_equal(sv[r:r + L], rv["scales"][a:a + L])
        assert gk[s].view(np.uint32) == np.float32(rk["g"]).view(np.uint32)
        assert gv[s].view(np.uint32) == np.float32(rv["g"]).view(np.uint32)
        assert np.array_equal(mk[s].view(np.uint32), rk["mean"].view(np.uint32))
    if len(fi) == 0:
        return 0
    rows = np.concatenate([np.arange(r, r + L) for r in fr])
    out_k = nv.kv_gather_dequant(pk, fr, fs, L, with_mean=True)
    out_v = nv.kv_gather_dequant(pv, fr, fs, L, with_mean=False)
    torch.cuda.synchronize()
    exp_k = oracle.kv_dequant(ck[rows], sk[rows], gk[fs], mean=mk[fs], tokens_per_group=L)
    exp_v = oracle.kv_dequant(cv[rows], sv[rows], gv[fs], tokens_per_group=L)
    assert same_bits_nan(bf16_bits(out_k), exp_k)
    assert same_bits_nan(bf16_bits(out_v), exp_v)
    return len(fi)


def run_events(nv, oracle, events, F, L, H, D, S_g, S_s, W, seed0):
    from nvfp4_block_quantization_gb300 import workloads as Wl

    cache = nv.KvCache(F, L, S_g, S_s, W)
    pk = nv.KvCachePool.allocate(cache, H, D, smooth=True)
    pv = nv.KvCachePool.allocate(cache, H, D, smooth=False)
    ws = nv.kv_workspace(F * L, H, D, 2)
    ref, sizes = {}, []
    for ev in events:
        if ev == "shot":
            cache.new_shot()
            continue
        sizes.append(check_view(nv, oracle, cache, pk, pv, ref, L))
        c = cache.n_chunks
        slot = cache.append()
        K = dev(Wl.to_bf16_bits(Wl.chunk_k(seed0 + 2 * c, T=F * L, H=H, D=D)))
        V = dev(Wl.to_bf16_bits(Wl.chunk_v(seed0 + 2 * c + 1, T=F * L, H=H, D=D)))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        outs = [pk.slot_outputs(cache, slot, status), pv.slot_outputs(cache, slot, status)]
        nv.kv_smooth_quant_batched([K, V], [True, False], workspace=ws, outs=outs, status=status)
        a, b = nv.kv_smooth_quant(K, True), nv.kv_smooth_quant(V, False)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref[c] = tuple(dict(codes=host(r.codes), scales=host(r.scales), g=float(host(r.tensor_scale)[0]),
                            mean=None if r.mean is None else host(r.mean)) for r in (a, b))
    sizes.append(check_view(nv, oracle, cache, pk, pv, ref, L))
    return sizes


def test_multi_shot_cache_small(nv, oracle):
    """Shot sink wider than a chunk, two prompt switches; frames of 16 tokens, 2 x 64 channels."""
    ev = ["a", "a", "a", "shot", "a", "a", "a", "shot", "a", "a", "a", "a"]
    sizes = run_events(nv, oracle, ev, F=4, L=16, H=2, D=64, S_g=2, S_s=5, W=6, seed0=700)
    assert sizes[0] == 0 and max(sizes) <= 2 + 5 + 6


def test_cache_read_sizes_full_frames(nv, oracle):
    """The cache-read workload's policy (3 sink + 18 rolling frames, 8-frame chunks) on full
    880-token frames of 24 x 128 channels: every view after the third chunk has 21 frames."""
    ev = ["a"] * 5
    sizes = run_events(nv, oracle, ev, F=8, L=880, H=24, D=128, S_g=3, S_s=3, W=18, seed0=900)
    assert sizes == [0, 8, 16, 21, 21, 21]


def test_gather_matches_plain_dequant(nv):
    """A view whose frames are one slot's chunk in order is that chunk's plain cache read."""
    from nvfp4_block_quantization_gb300 import workloads as Wl

    F, L, H, D = 4, 40, 3, 32
    cache = nv.KvCache(F, L, 0, 0, F)
    pool = nv.KvCachePool.allocate(cache, H, D, smooth=True)
    slot = cache.append()
    x = dev(Wl.to_bf16_bits(Wl.chunk_k(31, T=F * L, H=H, D=D)))
    o = pool.slot_outputs(cache, slot)
    nv.kv_smooth_quant(x, True, out=o)
    fi, fr, fs = cache.view()
    assert list(fi) == [0, 1, 2, 3]
    got = nv.kv_gather_dequant(pool, fr, fs, L, with_mean=True)
    want = nv.kv_dequant(o.codes, o.scales, o.tensor_scale, mean=o.mean)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
