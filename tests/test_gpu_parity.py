"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars:
  * codes, scales and the tensor scale bit-exact when both sides use the same
    mean (mean_in = the oracle's mean), and for every unsmoothed tensor;
  * end to end (GPU-computed mean): at most 1e-5 of blocks may differ, each by
    at most one code step in one element; dequantized values within 1e-3
    relative Frobenius error of the oracle's dequant;
  * dequant of the same codes bit-exact (NaN outputs compared as NaN).
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


def dev(a: np.ndarray):
    """numpy input (uint16 bf16 bits or float32) -> CUDA tensor of the same bytes."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def gpu_quant(nv, x, smooth, mean_in=None):
    mi = None if mean_in is None else torch.from_numpy(np.ascontiguousarray(mean_in, np.float32)).cuda()
    r = nv.kv_smooth_quant(dev(x), smooth, mean_in=mi)
    torch.cuda.synchronize()
    return dict(codes=host(r.codes), scales=host(r.scales), g=float(host(r.tensor_scale)[0]),
                mean=None if r.mean is None else host(r.mean), status=int(host(r.status)[0]))


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def nibbles(codes):
    c = codes.reshape(codes.shape[:-1] + (-1,))
    out = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.int64)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def signed_rank(code):
    return np.where(code & 8, -(code & 7), code & 7)


def assert_same_bits_f32(a, b):
    assert np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def compare_end_to_end(gpu, ref, D):
    """Return (#blocks differing, #blocks total); asserts each differing block is one code step in one element."""
    ga, ra = nibbles(gpu["codes"]), nibbles(ref["codes"])
    T, H = ga.shape[0], ga.shape[1]
    gb = ga.reshape(T, H, D // 16, 16)
    rb = ra.reshape(T, H, D // 16, 16)
    sdiff = gpu["scales"] != ref["scales"]
    cdiff = (gb != rb).any(axis=-1)
    bad = sdiff | cdiff
    for idx in zip(*np.nonzero(bad)):
        assert not sdiff[idx], f"block {idx}: scale {gpu['scales'][idx]} vs {ref['scales'][idx]}"
        d = np.abs(signed_rank(gb[idx]) - signed_rank(rb[idx]))
        assert (d > 0).sum() == 1 and d.max() == 1, f"block {idx}: codes {gb[idx]} vs {rb[idx]}"
    return int(bad.sum()), int(bad.size)


# ------------------------------------------------------------------ tiny config
def test_tiny_config_bit_exact(nv, oracle):
    from nvfp4_block_quantization_gb300 import workloads as W

    K, V = W.tiny_kv(0)
    for x, smooth in ((K, True), (V, False)):
        ref = oracle.kv_smooth_quant(x, smooth=smooth)
        got = gpu_quant(nv, x, smooth)
        assert got["status"] == 0 and ref["status"] == 0
        assert_same_bits_f32(got["g"], ref["g"])
        if smooth:
            assert_same_bits_f32(got["mean"], ref["mean"])
        assert np.array_equal(got["scales"], ref["scales"])
        assert np.array_equal(got["codes"], ref["codes"])
        # dequant, with and without the mean re-added
        for mean in ((None, ref["mean"]) if smooth else (None,)):
            rd = oracle.kv_dequant(ref["codes"], ref["scales"], ref["g"], mean=mean)
            gd = nv.kv_dequant(torch.from_numpy(ref["codes"]).cuda(), torch.from_numpy(ref["scales"]).cuda(),
                               torch.tensor([ref["g"]], dtype=torch.float32).cuda(),
                               mean=None if mean is None else torch.from_numpy(mean).cuda())
            assert np.array_equal(bf16_bits(gd), rd)


# ------------------------------------------------------------------ one chunk, full size
@pytest.fixture(scope="module")
def chunk():
    from nvfp4_block_quantization_gb300 import workloads as W

    return W.chunk_kv_bf16(2000, 2001)


@pytest.fixture(scope="module")
def chunk_ref(chunk, oracle):
    K, V = chunk
    return oracle.kv_smooth_quant(K, smooth=True), oracle.kv_smooth_quant(V, smooth=False)


def test_chunk_bit_exact_given_mean(nv, chunk, chunk_ref):
    K, V = chunk
    rk, rv = chunk_ref
    got = gpu_quant(nv, K, True, mean_in=rk["mean"])
    assert got["status"] == 0
    assert_same_bits_f32(got["g"], rk["g"])
    assert np.array_equal(got["scales"], rk["scales"])
    assert np.array_equal(got["codes"], rk["codes"])
    gv = gpu_quant(nv, V, False)
    assert_same_bits_f32(gv["g"], rv["g"])
    assert np.array_equal(gv["scales"], rv["scales"])
    assert np.array_equal(gv["codes"], rv["codes"])


def test_chunk_end_to_end(nv, chunk, chunk_ref, oracle):
    K, _ = chunk
    rk, _ = chunk_ref
    got = gpu_quant(nv, K, True)
    # the GPU mean is the oracle's (binary64 sum rounded once) in all but rare rounding cases
    mism = got["mean"].view(np.uint32).astype(np.int64) - rk["mean"].view(np.uint32).astype(np.int64)
    assert int((mism != 0).sum()) <= 3 and int(np.abs(mism).max()) <= 1
    nbad, nblk = compare_end_to_end(got, rk, 128)
    assert nbad <= 1e-5 * nblk, (nbad, nblk)
    # dequant (mean re-added) within 1e-3 relative Frobenius of the oracle's
    gd = nv.kv_dequant(torch.from_numpy(got["codes"]).cuda(), torch.from_numpy(got["scales"]).cuda(),
                       torch.tensor([got["g"]], dtype=torch.float32).cuda(), mean=torch.from_numpy(got["mean"]).cuda())
    rd = oracle.bf16_bits_to_f32(oracle.kv_dequant(rk["codes"], rk["scales"], rk["g"], mean=rk["mean"]))
    gdf = oracle.bf16_bits_to_f32(bf16_bits(gd)).astype(np.float64)
    rel = np.linalg.norm(gdf - rd) / np.linalg.norm(rd)
    assert rel <= 1e-3, rel


def test_chunk_batched_matches_reference(nv, chunk, chunk_ref):
    """K and V of one chunk in one batched enqueue -- the launch configuration the benchmark times."""
    K, V = chunk
    rk, rv = chunk_ref
    outs, status = nv.kv_smooth_quant_batched([dev(K), dev(V)], [True, False])
    torch.cuda.synchronize()
    assert int(host(status)[0]) == 0
    for o, r, sm in ((outs[0], rk, True), (outs[1], rv, False)):
        got = dict(codes=host(o.codes), scales=host(o.scales), g=float(host(o.tensor_scale)[0]))
        if sm:
            nbad, nblk = compare_end_to_end(got, r, 128)
            assert nbad <= 1e-5 * nblk
        else:
            assert np.array_equal(got["codes"], r["codes"]) and np.array_equal(got["scales"], r["scales"])
        assert_same_bits_f32(got["g"], r["g"])


# ------------------------------------------------------------------ shape sweep
SHAPES = [(1, 1, 16), (15, 1, 16), (16, 2, 32), (17, 3, 48), (64, 1, 64), (333, 5, 128), (7, 2, 3072),
          (1000, 24, 128)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("smooth", [True, False])
def test_shape_sweep(nv, oracle, shape, dtype, smooth):
    from nvfp4_block_quantization_gb300 import workloads as W

    T, H, D = shape
    seed = (T * 1000003 + H * 1009 + D * 7 + (dtype == "bf16") * 3 + int(smooth)) % 100000
    x = W.random_kv(seed, T, H, D, scale=2.0)
    if dtype == "bf16":
        x = W.to_bf16_bits(x)
    ref = oracle.kv_smooth_quant(x, smooth=smooth)
    got = gpu_quant(nv, x, smooth, mean_in=ref["mean"] if smooth else None)
    assert_same_bits_f32(got["g"], ref["g"])
    assert np.array_equal(got["scales"], ref["scales"])
    assert np.array_equal(got["codes"], ref["codes"])
    if smooth:
        e2e = gpu_quant(nv, x, smooth)
        mism = e2e["mean"].view(np.uint32).astype(np.int64) - ref["mean"].view(np.uint32).astype(np.int64)
        assert int((mism != 0).sum()) <= 3 and int(np.abs(mism).max()) <= 1
        nbad, nblk = compare_end_to_end(e2e, ref, D)
        assert nbad <= max(1, 1e-5 * nblk)


def test_empty_chunk(nv):
    x = torch.zeros((0, 2, 32), dtype=torch.bfloat16, device="cuda")
    r = nv.kv_smooth_quant(x, True)
    torch.cuda.synchronize()
    assert float(r.tensor_scale.item()) == 0.0 and int(r.status.item()) == 0
    assert np.array_equal(host(r.mean), np.zeros((2, 32), np.float32))


def test_all_zero_and_constant(nv, oracle):
    x = np.zeros((9, 2, 32), np.float32)
    got = gpu_quant(nv, x, False)
    assert got["g"] == 0.0 and not got["codes"].any() and not got["scales"].any()
    x = np.tile(np.arange(32, dtype=np.float32).reshape(1, 1, 32), (5, 3, 1))
    got = gpu_quant(nv, x, True)
    assert got["g"] == 0.0 and np.array_equal(got["mean"], x[0])


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
@pytest.mark.parametrize("smooth", [True, False])
def test_nonfinite_reported(nv, bad, smooth):
    x = np.ones((40, 2, 32), np.float32)
    x[17, 1, 5] = bad
    got = gpu_quant(nv, x, smooth)
    assert got["status"] == 1 and np.isnan(got["g"])
    assert np.all(got["scales"] == 0x7F) and not got["codes"].any()


def test_hand_row_on_gpu(nv, oracle):
    import json
    import os

    h = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.json")))
    x = np.concatenate([np.array(b["values"], dtype=np.float32) for b in h["blocks"]]).reshape(1, 1, 80)
    got = gpu_quant(nv, x, False)
    assert got["g"] == h["tensor"]["g"]
    assert got["scales"].ravel().tolist() == h["packed_row"]["scales"]
    assert got["codes"].ravel().tolist() == h["packed_row"]["codes"]


# ------------------------------------------------------------------ dequant
def test_dequant_groups_bit_exact(nv, oracle):
    from nvfp4_block_quantization_gb300 import workloads as W

    T, H, D, tpg = 3 * 40, 3, 64, 40
    parts = []
    for k in range(3):
        x = W.to_bf16_bits(W.random_kv(100 + k, tpg, H, D, scale=1.0 + k))
        parts.append(oracle.kv_smooth_quant(x, smooth=True))
    codes = np.concatenate([p["codes"] for p in parts])
    scales = np.concatenate([p["scales"] for p in parts])
    g = np.array([p["g"] for p in parts], np.float32)
    mean = np.stack([p["mean"] for p in parts])
    for m in (None, mean):
        rd = oracle.kv_dequant(codes, scales, g, mean=m, tokens_per_group=tpg)
        gd = nv.kv_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), torch.from_numpy(g).cuda(),
                           mean=None if m is None else torch.from_numpy(m).cuda(), tokens_per_group=tpg)
        assert np.array_equal(bf16_bits(gd), rd)
    # a mean array that is only 4-byte aligned (the kernel's scalar-load path)
    buf = torch.zeros(mean.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(mean.ravel()).cuda()
    m4 = buf[1:].view(mean.shape)
    assert m4.data_ptr() % 16 != 0
    gd = nv.kv_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), torch.from_numpy(g).cuda(),
                       mean=m4, tokens_per_group=tpg)
    assert np.array_equal(bf16_bits(gd), oracle.kv_dequant(codes, scales, g, mean=mean, tokens_per_group=tpg))


def test_dequant_nan_filler(nv, oracle):
    codes = np.zeros((2, 1, 16), np.uint8)
    scales = np.full((2, 1, 2), 0x7F, np.uint8)
    gd = nv.kv_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                       torch.tensor([np.nan], dtype=torch.float32).cuda())
    assert torch.isnan(gd.float()).all()


# ------------------------------------------------------------------ weights (2-D) and activations (1-D)
@pytest.mark.parametrize("shape", [(16, 16), (32, 48), (48, 80), (256, 512), (160, 3072)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_weight_2d_bit_exact(nv, oracle, shape, dtype):
    from nvfp4_block_quantization_gb300 import workloads as W

    M, N = shape
    w = W.weight(7, M, N)
    if dtype == "bf16":
        w = W.to_bf16_bits(w)
    ref = oracle.weight_quant_2d(w)
    r = nv.weight_quant_2d(dev(w))
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    assert_same_bits_f32(float(r.tensor_scale.item()), ref["g"])
    assert np.array_equal(host(r.scales), ref["scales"])
    assert np.array_equal(host(r.codes), ref["codes"])
    gd = nv.weight_dequant_2d(r.codes, r.scales, r.tensor_scale)
    assert np.array_equal(bf16_bits(gd), oracle.weight_dequant_2d(ref["codes"], ref["scales"], ref["g"]))


def test_weight_2d_full_size_sampled_tiles(nv, oracle):
    """3072 x 14336 weight: the tensor scale exactly, and 600 sampled tiles against the oracle's tile quantizer."""
    from nvfp4_block_quantization_gb300 import workloads as W

    M, N = 3072, 14336
    w = W.to_bf16_bits(W.weight(4, M, N))
    r = nv.weight_quant_2d(dev(w))
    torch.cuda.synchronize()
    wf = oracle.bf16_bits_to_f32(w)
    g = oracle.tensor_scale(float(np.abs(wf).max()))
    assert_same_bits_f32(float(r.tensor_scale.item()), g)
    scales, codes = host(r.scales), host(r.codes)
    rng = np.random.default_rng(0)
    for _ in range(600):
        ti, tj = int(rng.integers(M // 16)), int(rng.integers(N // 16))
        tile = wf[16 * ti:16 * ti + 16, 16 * tj:16 * tj + 16]
        d = oracle.block_detail(tile, g)
        assert scales[ti, tj] == d["scale"]
        got = nibbles(codes[16 * ti:16 * ti + 16, 8 * tj:8 * tj + 8]).ravel()
        assert np.array_equal(got, d["codes"].astype(np.int64))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_weight_2d_batched_bit_exact(nv, oracle, dtype):
    """Mixed shapes (one empty) in one batched call: every matrix matches the oracle on its own."""
    from nvfp4_block_quantization_gb300 import workloads as W

    shapes = [(256, 512), (0, 64), (48, 80), (160, 3072), (16, 16), (512, 256)]
    ws_np = [W.weight(20 + i, M, N) for i, (M, N) in enumerate(shapes)]
    if dtype == "bf16":
        ws_np = [W.to_bf16_bits(w) for w in ws_np]
    outs, status = nv.weight_quant_2d_batched([dev(w) for w in ws_np])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for w, o in zip(ws_np, outs):
        if w.shape[0] == 0:
            assert float(o.tensor_scale.item()) == 0.0
            continue
        ref = oracle.weight_quant_2d(w)
        assert_same_bits_f32(float(o.tensor_scale.item()), ref["g"])
        assert np.array_equal(host(o.scales), ref["scales"])
        assert np.array_equal(host(o.codes), ref["codes"])


def test_weight_2d_batched_all_empty(nv):
    """A batch of empty matrices writes tensor scale 0 and status 0."""
    ws = [torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")]
    outs, status = nv.weight_quant_2d_batched(ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert all(float(o.tensor_scale.item()) == 0.0 for o in outs)


def test_weight_2d_batched_many_and_nonfinite(nv):
    """70 matrices (two launch pairs of at most 64) equal the single calls; a NaN in the first sets the shared status."""
    from nvfp4_block_quantization_gb300 import workloads as W

    shapes = [(16 * (1 + i % 5), 16 * (1 + (3 * i) % 7)) for i in range(70)]
    ws = [dev(W.to_bf16_bits(W.weight(100 + i, M, N))) for i, (M, N) in enumerate(shapes)]
    ws[0][3, 5] = float("nan")
    outs, status = nv.weight_quant_2d_batched(ws)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    assert torch.isnan(outs[0].tensor_scale).all()
    assert bool((outs[0].scales == 0x7F).all()) and bool((outs[0].codes == 0).all())
    for w, o in zip(ws[1:], outs[1:]):
        s = nv.weight_quant_2d(w)
        torch.cuda.synchronize()
        assert int(s.status.item()) == 0
        assert torch.equal(o.codes, s.codes) and torch.equal(o.scales, s.scales)
        assert torch.equal(o.tensor_scale.view(torch.int32), s.tensor_scale.view(torch.int32))
    # clean batches after the NaN one, twice on one workspace and the same status word: no
    # error, and the same bits (the workspace returns to zero after every call)
    ws2 = ws[1:]
    wsp = nv.w2d_batched_workspace(len(ws2))
    for _ in range(2):
        outs2, status2 = nv.weight_quant_2d_batched(ws2, workspace=wsp, status=status)
        torch.cuda.synchronize()
        assert int(status2.item()) == 0
        for o2, o in zip(outs2, outs[1:]):
            assert torch.equal(o2.codes, o.codes) and torch.equal(o2.scales, o.scales)
            assert torch.equal(o2.tensor_scale.view(torch.int32), o.tensor_scale.view(torch.int32))
    assert not bool(wsp.any())


def test_activations_1d_bit_exact(nv, oracle):
    from nvfp4_block_quantization_gb300 import workloads as W

    a = W.to_bf16_bits(W.activations()).reshape(7040, 1, 3072)
    ref = oracle.kv_smooth_quant(a, smooth=False)
    got = gpu_quant(nv, a, False)
    assert_same_bits_f32(got["g"], ref["g"])
    assert np.array_equal(got["scales"], ref["scales"])
    assert np.array_equal(got["codes"], ref["codes"])


# ------------------------------------------------------------------ batched = single
def test_batched_equals_single_calls(nv):
    from nvfp4_block_quantization_gb300 import workloads as W

    xs, flags = [], []
    for layer in range(3):
        sk, sv = W.layer_seeds(layer)
        xs += [dev(W.to_bf16_bits(W.chunk_k(sk, T=880, H=4, D=128))), dev(W.to_bf16_bits(W.chunk_v(sv, T=880, H=4, D=128)))]
        flags += [True, False]
    outs, status = nv.kv_smooth_quant_batched(xs, flags)
    torch.cuda.synchronize()
    for x, f, o in zip(xs, flags, outs):
        s = nv.kv_smooth_quant(x, f)
        torch.cuda.synchronize()
        assert torch.equal(o.codes, s.codes) and torch.equal(o.scales, s.scales)
        assert torch.equal(o.tensor_scale, s.tensor_scale)
        if f:
            assert torch.equal(o.mean, s.mean)


# ------------------------------------------------------------------ split passes
def test_split_passes_match_combined(nv):
    """kv_stats_batched + kv_quant_batched give the combined call's bits, also across two streams."""
    from nvfp4_block_quantization_gb300 import workloads as W

    Kb, Vb = W.chunk_kv_bf16(2000, 2001)
    K, V = dev(Kb[:1000]), dev(Vb[:1000])
    T, H, D = K.shape
    ref, st = nv.kv_smooth_quant_batched([K, V], [True, False])
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    def fresh(smooth_flags):
        outs, status = [], torch.zeros(1, dtype=torch.int32, device="cuda")
        for sm in smooth_flags:
            outs.append(nv.KvQuantized(torch.empty((T, H, D // 2), dtype=torch.uint8, device="cuda"),
                                       torch.empty((T, H, D // 16), dtype=torch.uint8, device="cuda"),
                                       torch.empty(1, dtype=torch.float32, device="cuda"),
                                       torch.empty((H, D), dtype=torch.float32, device="cuda") if sm else None,
                                       status))
        return outs, status

    def same(a, b):
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
        assert torch.equal(a.tensor_scale.view(torch.int32), b.tensor_scale.view(torch.int32))
        if a.mean is not None:
            assert torch.equal(a.mean.view(torch.int32), b.mean.view(torch.int32))

    # same batch, two enqueues, twice on one workspace
    ws = nv.kv_workspace(T, H, D, 2)
    for _ in range(2):
        outs, status = fresh([True, False])
        nv.kv_stats_batched([K, V], [True, False], ws, outs)
        nv.kv_quant_batched([K, V], [True, False], ws, outs, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        same(outs[0], ref[0])
        same(outs[1], ref[1])

    # K and V as separate one-job batches on two streams: V's statistics run beside K's quantization
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    wk, wv = nv.kv_workspace(T, H, D, 1), nv.kv_workspace(T, H, D, 1)
    ok_, sk = fresh([True])
    ov, sv = fresh([False])
    for _ in range(2):
        with torch.cuda.stream(s1):
            nv.kv_stats_batched([K], [True], wk, ok_, stream=s1)
            nv.kv_quant_batched([K], [True], wk, ok_, sk, stream=s1)
        with torch.cuda.stream(s2):
            nv.kv_stats_batched([V], [False], wv, ov, stream=s2)
            nv.kv_quant_batched([V], [False], wv, ov, sv, stream=s2)
        torch.cuda.synchronize()
        assert int(sk.item()) == 0 and int(sv.item()) == 0
        same(ok_[0], ref[0])
        same(ov[0], ref[1])
