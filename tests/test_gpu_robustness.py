"""GPU checks beyond the parity sweeps: the conversion instructions against the
oracle's encoders over a dense sweep of fp32 inputs, a bounded wait that runs
out, and batches of many tensors (one and two launch groups).

The conversions are the steps every quantizer's bit-exactness rests on:
round-to-nearest-even E2M1 codes with saturation at 6 and the sign kept, and
E4M3 block scales rounded to nearest even and saturated at 448 (the NVFP4
definition the quantizers implement).
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


def _near(values, ulps=64):
    """Every fp32 within +-ulps of each value (both signs)."""
    v = np.asarray(values, dtype=np.float32).view(np.int32).astype(np.int64)
    off = np.arange(-ulps, ulps + 1, dtype=np.int64)
    bits = (v[:, None] + off[None, :]).reshape(-1)
    bits = bits[(bits >= 0) & (bits < 0x7F800000)].astype(np.int32)
    f = bits.view(np.float32)
    return np.concatenate([f, -f])


def _sweep_inputs():
    rng = np.random.default_rng(7)
    parts = []
    # random bit patterns over the whole fp32 range (NaNs excluded)
    r = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    parts.append(r[~np.isnan(r)])
    # dense: exponents 2^-14 .. 2^10, every 128th mantissa, both signs
    e = np.arange(127 - 14, 127 + 11, dtype=np.uint32)
    m = np.arange(0, 1 << 23, 128, dtype=np.uint32)
    d = ((e[:, None] << 23) | m[None, :]).reshape(-1).view(np.float32)
    parts += [d, -d]
    # every E2M1 rounding midpoint (ties go to the even code) and the saturation edge
    parts.append(_near([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0]))
    # every E4M3 midpoint between consecutive finite codes, and around 448 / 464
    vals = np.array([float(np.float32(v)) for v in _e4m3_values()], dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2.0
    parts.append(_near(np.concatenate([mids, [448.0, 464.0, 2.0 ** -10, 2.0 ** -9]])))
    # specials
    parts.append(np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4028235e38, -3.4028235e38], np.float32))
    return np.ascontiguousarray(np.concatenate(parts).astype(np.float32))


def _e4m3_values():
    """The 127 non-negative finite E4M3 values in code order, from the format's definition."""
    out = []
    for c in range(0x7F):
        e, mm = c >> 3, c & 7
        out.append(mm * 2.0 ** -9 if e == 0 else (1 + mm / 8.0) * 2.0 ** (e - 7))
    return out


def test_conversion_instructions_match_the_oracle(nv, oracle):
    x = _sweep_inputs()
    e2m1, e4m3, dec, val = nv.selftest_cvt(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    e2m1 = e2m1.cpu().numpy()
    e4m3 = e4m3.cpu().numpy().view(np.uint16)
    want2 = oracle.e2m1_encode_array(x)
    want4 = oracle.e4m3_encode_array(x)
    bad2 = np.nonzero(((e2m1 & 0xF) != want2) | ((e2m1 >> 4) != want2))[0]
    assert bad2.size == 0, f"E2M1 codes differ at {x[bad2[:5]]}: got {e2m1[bad2[:5]]}, want {want2[bad2[:5]]}"
    bad4 = np.nonzero(((e4m3 & 0xFF) != want4) | ((e4m3 >> 8) != want4))[0]
    assert bad4.size == 0, f"E4M3 codes differ at {x[bad4[:5]]}: got {e4m3[bad4[:5]]}, want {want4[bad4[:5]]}"
    # decodes: every byte as two E2M1 codes (f16 pair), every E4M3 code as fp32
    dec = dec.cpu().numpy().view(np.uint32)
    for b in range(256):
        lo = np.array([dec[b] & 0xFFFF], np.uint16).view(np.float16)[0]
        hi = np.array([dec[b] >> 16], np.uint16).view(np.float16)[0]
        for got, code in ((lo, b & 0xF), (hi, b >> 4)):
            want = np.float16(oracle.e2m1_decode(code))
            assert np.array_equal(np.array([got]).view(np.uint16), np.array([want]).view(np.uint16)), (b, code)
    val = val.cpu().numpy()
    for b in range(256):
        want = oracle.e4m3_decode(b)
        if np.isnan(want):
            assert np.isnan(val[b]), b
        else:
            assert np.float32(val[b]).view(np.uint32) == np.float32(want).view(np.uint32), (b, val[b], want)


def test_quantization_wait_runs_out(nv, oracle):
    """A quantization pass enqueued on a clean workspace without its statistics pass
    waits (bounded, about 2 s) for statistics that never come, then reports
    NVFP4_DEV_TIMEOUT and writes the filler outputs; a zero-filled workspace then
    serves a normal call."""
    from nvfp4_block_quantization_gb300 import workloads as W

    K = W.to_bf16_bits(W.random_kv(11, 64, 2, 64))
    x = torch.from_numpy(K.view(np.int16)).view(torch.bfloat16).cuda()
    outs, status = nv.kv_smooth_quant_batched([x], [True])  # allocates outputs, workspace-free run
    ws = nv.kv_workspace(64, 2, 64, 1, x.device)
    ws.zero_()
    nv.kv_quant_batched([x], [True], ws, outs, status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & nv._lib.NVFP4_DEV_TIMEOUT, st
    assert bool((outs[0].scales == 0x7F).all()) and bool((outs[0].codes == 0).all())
    assert np.isnan(float(outs[0].tensor_scale.item()))
    # the documented recovery: zero-fill the workspace, then the call works again
    ws.zero_()
    outs2, status2 = nv.kv_smooth_quant_batched([x], [True], workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.kv_smooth_quant(K, smooth=True)
    assert int(status2.item()) == 0
    assert np.array_equal(outs2[0].scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(outs2[0].codes.cpu().numpy(), ref["codes"])


@pytest.mark.parametrize("n_jobs", [60, 70])
def test_many_tensor_batch_matches_the_oracle(nv, oracle, n_jobs):
    """60 tensors (one layer-stack chunk write: K and V of 30 layers, one launch group)
    and 70 (two launch groups), K smoothed and V not, each with its own seed."""
    from nvfp4_block_quantization_gb300 import workloads as W

    T, H, D = 48, 2, 64
    xs_np, flags = [], []
    for j in range(n_jobs):
        smooth = j % 2 == 0
        a = W.random_kv(4000 + j, T, H, D, offset_sd=3.0 if smooth else 0.0)
        xs_np.append(W.to_bf16_bits(a))
        flags.append(smooth)
    xs = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda() for a in xs_np]
    outs, status = nv.kv_smooth_quant_batched(xs, flags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for j in range(n_jobs):
        ref = oracle.kv_smooth_quant(xs_np[j], smooth=flags[j])
        o = outs[j]
        assert np.float32(o.tensor_scale.item()).view(np.uint32) == np.float32(ref["g"]).view(np.uint32), j
        if flags[j]:
            assert np.array_equal(o.mean.cpu().numpy().view(np.uint32), ref["mean"].view(np.uint32)), j
        assert np.array_equal(o.scales.cpu().numpy(), ref["scales"]), j
        assert np.array_equal(o.codes.cpu().numpy(), ref["codes"]), j


def test_headroom_tensor_scale_matches_the_oracle(nv, oracle):
    """g = amax / 1792 (every block's 4-candidate under 448): codes, scales and g
    bit-exact against the oracle's headroom statement, K smoothed and V not."""
    from nvfp4_block_quantization_gb300 import workloads as W

    K, V = W.tiny_kv(0)
    Kb = W.to_bf16_bits(W.random_kv(21, 96, 3, 64))
    for arrays in ((K, V), (Kb, W.to_bf16_bits(W.random_kv(22, 96, 3, 64, offset_sd=0.0)))):
        xs = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda() if a.dtype == np.uint16
              else torch.from_numpy(a).cuda() for a in arrays]
        outs, status = nv.kv_smooth_quant_batched(xs, [True, False], headroom=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for a, smooth, o in zip(arrays, (True, False), outs):
            ref = oracle.kv_smooth_quant(a, smooth=smooth, headroom=True)
            assert np.float32(o.tensor_scale.item()).view(np.uint32) == np.float32(ref["g"]).view(np.uint32)
            assert np.array_equal(o.scales.cpu().numpy(), ref["scales"])
            assert np.array_equal(o.codes.cpu().numpy(), ref["codes"])
            # the amax block can now pick 4: with the standard scale it never does
            std = oracle.kv_smooth_quant(a, smooth=smooth)
            assert not np.array_equal(std["scales"], ref["scales"])
