"""GPU: attention over the NVFP4 cache (nvfp4_kv_attention_decode) against the oracle.

Chunks are quantized into pool slots by the cache manager and the quantizer; queries
attend over each chunk's view.  The GPU evaluates scores and the softmax in fp32: per
lane and 16-channel block, a fused chain over q . Q_k, times the block scale, plus the
slot's q . mean (itself a 16-term chain); a shuffle tree over the token's lanes; an online
softmax per split of 256 to 2048 tokens (each lane group's fp32 sums of at most 128 terms);
then exact merging.  So each output obeys
    |o - o_ref| <= Vmax * (64 * 2^-24 * A + 1e-5)
with A = max_t |scale| sum_d |q_d| (|Q S|_td + |mean_d|) and Vmax = max |v| of the head,
both from the oracle: a score error of at most about 23 units of 2^-24 relative to A moves
each softmax weight by at most twice that, and 1e-5 covers the fast exponential and the
fp32 sums of at most a few hundred terms.
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


def fill_cache(nv, F, L, H, D, S_g, S_s, W, n_chunks, shot_after=None, seed0=1200):
    from nvfp4_block_quantization_gb300 import workloads as Wl

    cache = nv.KvCache(F, L, S_g, S_s, W)
    pk = nv.KvCachePool.allocate(cache, H, D, smooth=True)
    pv = nv.KvCachePool.allocate(cache, H, D, smooth=False)
    for c in range(n_chunks):
        if shot_after is not None and c == shot_after:
            cache.new_shot()
        slot = cache.append()
        K = dev(Wl.to_bf16_bits(Wl.chunk_k(seed0 + 2 * c, T=F * L, H=H, D=D)))
        V = dev(Wl.to_bf16_bits(Wl.chunk_v(seed0 + 2 * c + 1, T=F * L, H=H, D=D)))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        nv.kv_smooth_quant_batched([K, V], [True, False],
                                   outs=[pk.slot_outputs(cache, slot, st), pv.slot_outputs(cache, slot, st)], status=st)
    torch.cuda.synchronize()
    return cache, pk, pv


def reference(oracle_attn, cache, pk, pv, q, scale):
    fi, fr, fs = cache.view()
    L = cache.state.tokens_per_frame
    rows = np.concatenate([np.arange(r, r + L) for r in fr])
    slot_of = np.repeat(fs, L)
    mean = host(pk.mean)[slot_of]
    k0 = oracle_attn.dequant_fp32(host(pk.codes)[rows], host(pk.scales)[rows], host(pk.g)[slot_of])
    k = oracle_attn.dequant_fp32(host(pk.codes)[rows], host(pk.scales)[rows], host(pk.g)[slot_of], mean)
    v = oracle_attn.dequant_fp32(host(pv.codes)[rows], host(pv.scales)[rows], host(pv.g)[slot_of])
    out, _, Vmax = oracle_attn.attention_decode(q, k, v, scale)
    # the scale of the score's rounding: |scale| sum_d |q_d| (|Q S| + |mean|), worst token
    parts = np.abs(k0.astype(np.float64)) + np.abs(mean.astype(np.float64))
    A = np.einsum("ihd,thd->iht", np.abs(q.astype(np.float64)), parts).max(axis=2) * abs(scale)
    return fr, fs, out, A, Vmax


def check(out, ref, A, Vmax):
    tol = Vmax[None, :, None] * (64 * 2.0 ** -24 * A[:, :, None] + 1e-5)
    bad = np.abs(out - ref) > tol
    assert not bad.any(), (int(bad.sum()), float((np.abs(out - ref) - tol).max()))


@pytest.mark.parametrize("n_q", [1, 2, 3, 4])
def test_attention_small_multi_shot(nv, n_q):
    """Frames of 16 tokens, 2 heads x 64 channels, a shot switch: the view mixes slots."""
    from oracle import attention as oa

    cache, pk, pv = fill_cache(nv, F=4, L=16, H=2, D=64, S_g=2, S_s=5, W=6, n_chunks=7, shot_after=3)
    q = np.random.default_rng(n_q).standard_normal((n_q, 2, 64)).astype(np.float32)
    scale = 64 ** -0.5
    fr, fs, ref, A, Vmax = reference(oa, cache, pk, pv, q, scale)
    out = host(nv.kv_attention_decode(torch.from_numpy(q).cuda(), pk, pv, fr, fs, 16, scale))
    check(out, ref, A, Vmax)


def test_attention_cache_read_view(nv):
    """The cache-read workload's view: 3 sink + 18 rolling frames of 880 tokens, 24 heads x 128."""
    from oracle import attention as oa

    cache, pk, pv = fill_cache(nv, F=8, L=880, H=24, D=128, S_g=3, S_s=3, W=18, n_chunks=5)
    q = (np.random.default_rng(9).standard_normal((2, 24, 128)) * 0.5).astype(np.float32)
    scale = 128 ** -0.5
    fr, fs, ref, A, Vmax = reference(oa, cache, pk, pv, q, scale)
    assert len(fr) == 21
    out = host(nv.kv_attention_decode(torch.from_numpy(q).cuda(), pk, pv, fr, fs, 880, scale))
    check(out, ref, A, Vmax)
