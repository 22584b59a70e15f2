"""GPU: attention of a block of queries over the NVFP4 cache on the tensor cores
(nvfp4_kv_attention_prefill) against the oracle.

The kernel multiplies bf16 queries by K' = Q E_k (exact in bf16) on the tensor cores with fp32
sums, forms s = scale (g_k (q . K') + q . mean) in fp32, and accumulates the output from
P' = bf16(exp(s - m) g_v / G) times V' = Q E_v (exact) in fp32.  Against the binary64 oracle
(keys and values dequantized in fp32 as the cache read defines them) each output obeys
    |o - o_ref| <= 2^-8 B + 2 eps (B + |o_ref|) + (n_keys + 4) 2^-23 (B + |o_ref|) + 1e-7
with B = sum_t p_t |v_t| (oracle) and eps = 160 * 2^-24 * A,
A = max_t |scale| sum_d |q_d| (|Q S|_td + |mean_d|):
- rounding P' to bf16 changes each weight by at most 2^-9 relative (2^-8 B with the margin of
  the fp32 product before it);
- the score's fp32 sums (128 products, the mean's 128-term chain, the oracle's own fp32
  dequant roundings) stay within about 136 units of 2^-24 A, and a score error eps moves each
  normalised weight by at most about 2 eps;
- the fp32 sums over n_keys weights (l, and the tensor cores' accumulation of P' V') and the
  final G O / l add at most (n_keys + 4) 2^-23 relative.
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


def fill_cache(nv, F, L, H, D, S_g, S_s, W, n_chunks, shot_after=None, seed0=1400, k_gains=None):
    from nvfp4_block_quantization_gb300 import workloads as Wl

    cache = nv.KvCache(F, L, S_g, S_s, W)
    pk = nv.KvCachePool.allocate(cache, H, D, smooth=True)
    pv = nv.KvCachePool.allocate(cache, H, D, smooth=False)
    for c in range(n_chunks):
        if shot_after is not None and c == shot_after:
            cache.new_shot()
        slot = cache.append()
        gain = 1.0 if k_gains is None else k_gains[c]
        K = dev(Wl.to_bf16_bits(Wl.chunk_k(seed0 + 2 * c, T=F * L, H=H, D=D) * np.float32(gain)))
        V = dev(Wl.to_bf16_bits(Wl.chunk_v(seed0 + 2 * c + 1, T=F * L, H=H, D=D)))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        nv.kv_smooth_quant_batched([K, V], [True, False],
                                   outs=[pk.slot_outputs(cache, slot, st), pv.slot_outputs(cache, slot, st)], status=st)
    torch.cuda.synchronize()
    return cache, pk, pv


def queries(n_q, H, D, seed, sd=1.0):
    from nvfp4_block_quantization_gb300 import workloads as Wl

    bits = Wl.to_bf16_bits((np.random.default_rng(seed).standard_normal((n_q, H, D)) * sd).astype(np.float32))
    return bits, (bits.astype(np.uint32) << 16).view(np.float32)


def run_and_check(nv, cache, pk, pv, qbits, qf, scale, heads=None, rows_q=None, split=True):
    """Runs all queries on the GPU (with the last wave's units split along the keys when
    `split`); compares the oracle on `heads` (all by default) and on the query rows `rows_q`
    (all by default)."""
    from oracle import attention as oa

    fi, fr, fs = cache.view()
    L = cache.state.tokens_per_frame
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = host(nv.kv_attention_prefill(dev(qbits), pk, pv, fr, fs, L, scale, status=status, split=split))
    assert int(host(status)[0]) == 0
    if rows_q is not None:
        out, qf = out[rows_q], qf[rows_q]
    heads = list(range(qf.shape[1])) if heads is None else heads
    rows = np.concatenate([np.arange(r, r + L) for r in fr])
    slot_of = np.repeat(fs, L)
    n_keys = rows.size
    for h in heads:
        sl = slice(h, h + 1)
        mean = host(pk.mean)[slot_of][:, sl]
        k0 = oa.dequant_fp32(host(pk.codes)[rows][:, sl], host(pk.scales)[rows][:, sl], host(pk.g)[slot_of])
        k = oa.dequant_fp32(host(pk.codes)[rows][:, sl], host(pk.scales)[rows][:, sl], host(pk.g)[slot_of], mean)
        v = oa.dequant_fp32(host(pv.codes)[rows][:, sl], host(pv.scales)[rows][:, sl], host(pv.g)[slot_of])
        ref, B = oa.attention_weighted_abs(qf[:, sl], k, v, scale)
        parts = np.abs(k0.astype(np.float64)) + np.abs(mean.astype(np.float64))
        A = np.einsum("ihd,thd->iht", np.abs(qf[:, sl].astype(np.float64)), parts).max(axis=2) * abs(scale)
        eps = 160 * 2.0 ** -24 * A[:, :, None]
        tol = (2.0 ** -8 * B + 2 * eps * (B + np.abs(ref)) + (n_keys + 4) * 2.0 ** -23 * (B + np.abs(ref)) + 1e-7)
        err = np.abs(out[:, sl].astype(np.float64) - ref)
        bad = err > tol
        assert not bad.any(), (h, int(bad.sum()), float((err - tol).max()), float(err.max()))


def test_prefill_small_multi_shot(nv):
    """Frames of 16 tokens, 2 heads x 128 channels, a shot switch (the view mixes slots);
    200 queries: one full 128-query tile and a ragged one; the last key tile is ragged."""
    cache, pk, pv = fill_cache(nv, F=4, L=16, H=2, D=128, S_g=2, S_s=5, W=6, n_chunks=7, shot_after=3)
    qbits, qf = queries(200, 2, 128, 3)
    run_and_check(nv, cache, pk, pv, qbits, qf, 128 ** -0.5)


def test_prefill_one_query_and_one_frame(nv):
    """The smallest case: one query, a view of one 16-token frame."""
    cache, pk, pv = fill_cache(nv, F=1, L=16, H=1, D=128, S_g=1, S_s=1, W=1, n_chunks=1)
    qbits, qf = queries(1, 1, 128, 4)
    run_and_check(nv, cache, pk, pv, qbits, qf, 0.3)


@pytest.mark.parametrize("split", [True, False])
def test_prefill_cache_read_view(nv, split):
    """The cache-read workload's view: 3 sink + 18 rolling frames of 880 tokens, 24 heads x 128,
    130 queries (one 256-query unit per head, so all 24 units form the last wave and are split along
    the keys unless `split` is off); heads 0, 11 and 23 against the oracle."""
    cache, pk, pv = fill_cache(nv, F=8, L=880, H=24, D=128, S_g=3, S_s=3, W=18, n_chunks=5)
    assert len(cache.view()[1]) == 21
    qbits, qf = queries(130, 24, 128, 9, sd=0.5)
    run_and_check(nv, cache, pk, pv, qbits, qf, 128 ** -0.5, heads=[0, 11, 23], split=split)


def test_prefill_whole_chunk_sampled(nv):
    """The row's shape: a whole chunk of 7040 queries x 24 heads over the 21-frame view in one call;
    48 sampled query rows (both halves of many CTAs, the last ragged CTA included) of heads 5, 17
    and 23 against the oracle (on 152 SMs the last 64 of the 672 units, heads 21-23, run split)."""
    cache, pk, pv = fill_cache(nv, F=8, L=880, H=24, D=128, S_g=3, S_s=3, W=18, n_chunks=5, seed0=1500)
    qbits, qf = queries(7040, 24, 128, 11, sd=0.5)
    rows_q = np.sort(np.concatenate([np.random.default_rng(12).choice(7040, 44, replace=False),
                                     np.array([0, 255, 256, 7039])]))
    run_and_check(nv, cache, pk, pv, qbits, qf, 128 ** -0.5, heads=[5, 17, 23], rows_q=rows_q)


@pytest.mark.parametrize("split", [True, False])
def test_prefill_rising_scores(nv, split):
    """K of later chunks scaled up (gains 1/4, 1, 4, 16, 64): the scores jump by far more than the
    lazy-rescale step at chunk boundaries, so the running maximum moves mid-view and O is rescaled
    in TMEM; with the key split the two halves' maxima differ by orders of magnitude, so the merge
    weights are near 0 and 1.  16 frames of 64 tokens, 2 heads, 300 queries."""
    cache, pk, pv = fill_cache(nv, F=4, L=64, H=2, D=128, S_g=2, S_s=2, W=12, n_chunks=5,
                               k_gains=[0.25, 1.0, 4.0, 16.0, 64.0])
    qbits, qf = queries(300, 2, 128, 21)
    run_and_check(nv, cache, pk, pv, qbits, qf, 128 ** -0.5, split=split)

