"""GPU: the W4A4 NVFP4 GEMM through the C ABI against the oracle reference.

Operands come from this library's quantizers (1-D activation blocks, 16x16 weight
tiles), whose bits are checked against the oracle elsewhere.  The GPU sums exact
products in fp32 on the tensor cores and rounds the scaled result to bf16, so each
output must satisfy
    |y - ref| <= 2^-8 |ref| + (1 + 2^-8) * 2 K 2^-24 * sum_k |x w| * gX gW
(bf16 rounding of the result, plus the worst case of an fp32 summation of K
terms, doubled), with ref and the absolute sum from the oracle in binary64.
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


def bf16_dev(a: np.ndarray):
    from nvfp4_block_quantization_gb300 import workloads as W

    return torch.from_numpy(W.to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    return t.detach().cpu().numpy()


def quantized_operands(nv, X, Wm):
    M, K = X.shape
    xq = nv.kv_smooth_quant(bf16_dev(X).view(M, 1, K), False)
    wq = nv.weight_quant_2d(bf16_dev(Wm))
    torch.cuda.synchronize()
    assert int(host(xq.status)[0]) == 0 and int(host(wq.status)[0]) == 0
    return xq, wq


def run_gemm(nv, xq, wq, M, N, K):
    xs = nv.mma_scales(xq.scales.view(M, K // 16), K)
    ws = nv.mma_scales(wq.scales, K, tile2d=True)
    plan = nv.GemmPlan(M, N, K)
    work = nv.gemm_workspace()  # zeroed: its first int32 is the kernel's bounded-wait error flag
    y = nv.gemm_w4a4(plan, xq.codes.view(M, K // 2), xs, xq.tensor_scale, wq.codes, ws, wq.tensor_scale, work)
    torch.cuda.synchronize()
    assert int(work[:4].view(torch.int32).item()) == 0
    return y.float().cpu().numpy().astype(np.float64)


def check(y, ref, sabs, K):
    tol = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * 2 * K * 2.0 ** -24 * sabs
    bad = np.abs(y - ref) > tol
    assert not bad.any(), (int(bad.sum()), float(np.max(np.abs(y - ref) - tol)))


def test_scale_layout_matches_its_definition(nv):
    """Block (r, c) lands in tile (r / 128, c / 4) at (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4;
    the padding is zero; a weight tile's scale covers its 16 rows."""
    rng = np.random.default_rng(3)
    rows, K = 300, 16 * 13
    KB = K // 16
    s = rng.integers(1, 255, size=(rows, KB), dtype=np.uint8)
    got = host(nv.mma_scales(torch.from_numpy(s).cuda(), K))
    kbt = (KB + 3) // 4
    want = np.zeros(((rows + 127) // 128) * 128 * kbt * 4, np.uint8)
    for r in range(rows):
        for c in range(KB):
            want[((r // 128) * kbt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4] = s[r, c]
    assert np.array_equal(got[:want.size], want)
    t = rng.integers(1, 255, size=(rows // 16 + 1, KB), dtype=np.uint8)
    got2 = host(nv.mma_scales(torch.from_numpy(t).cuda(), K, tile2d=True))
    rows2 = t.shape[0] * 16
    want2 = np.zeros(((rows2 + 127) // 128) * 128 * kbt * 4, np.uint8)
    for r in range(rows2):
        for c in range(KB):
            want2[((r // 128) * kbt + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4] = t[r // 16, c]
    assert np.array_equal(got2[:want2.size], want2)


def test_w4a4_small_ragged(nv):
    """M = 200 (not a multiple of the 128-row scale tile), N = 384, K = 512."""
    from oracle import gemm as og

    rng = np.random.default_rng(11)
    M, N, K = 200, 384, 512
    X = rng.standard_normal((M, K)).astype(np.float32)
    Wm = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Wm.flat[rng.choice(Wm.size, Wm.size // 1000, replace=False)] *= 30.0
    xq, wq = quantized_operands(nv, X, Wm)
    y = run_gemm(nv, xq, wq, M, N, K)
    ref, sabs = og.gemm_w4a4(host(xq.codes).reshape(M, K // 2), host(xq.scales).reshape(M, K // 16),
                             float(host(xq.tensor_scale)[0]), host(wq.codes), host(wq.scales),
                             float(host(wq.tensor_scale)[0]))
    check(y, ref, sabs, K)


@pytest.mark.parametrize("M,N,K", [(300, 48, 96), (129, 272, 320), (1, 16, 32), (385, 512, 768), (200, 400, 512)])
def test_w4a4_tails(nv, M, N, K):
    """Edges of the 128 x 256 output tiles and of the 256-element K slices: N = 16 past a tile
    boundary, K not a multiple of 64 (a half-filled last MMA step), M = 1, an odd number of row
    tiles; every output against the oracle.  With few tiles the whole grid is one last wave: at
    N = 512 and 400 every tile runs as two 128-column halves on two CTAs (at N = 400 the last
    halves are 128 and 16 columns wide); tiles of at most 128 valid columns (N = 48, 16, 272 - 256)
    keep the grid whole."""
    from oracle import gemm as og

    rng = np.random.default_rng(M + N + K)
    X = rng.standard_normal((M, K)).astype(np.float32)
    Wm = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xq, wq = quantized_operands(nv, X, Wm)
    y = run_gemm(nv, xq, wq, M, N, K)
    ref, sabs = og.gemm_w4a4(host(xq.codes).reshape(M, K // 2), host(xq.scales).reshape(M, K // 16),
                             float(host(xq.tensor_scale)[0]), host(wq.codes), host(wq.scales),
                             float(host(wq.tensor_scale)[0]))
    check(y, ref, sabs, K)


def test_w4a4_linear_sizes_sampled_rows(nv):
    """Activations 7040 x 3072 ~ N(0, 1) and a 3072 x 3072 weight ~ N(0, 0.02^2) with 0.1% x30,
    as the GEMM of a W4A4 linear layer; 64 sampled rows and 4 chosen ones against the oracle (on
    152 SMs the last 52 of the 660 tiles run as 128-column halves: rows 6400-6527 from column 2048
    on, and every row from 6528)."""
    from nvfp4_block_quantization_gb300 import workloads as W
    from oracle import gemm as og

    M, N, K = 7040, 3072, 3072
    X = W.activations(T=M, D=K)
    Wm = W.weight(0, N, K)
    xq, wq = quantized_operands(nv, X, Wm)
    y = run_gemm(nv, xq, wq, M, N, K)
    rows = np.sort(np.concatenate([np.random.default_rng(5).choice(M, 64, replace=False),
                                   np.array([6400, 6527, 6528, 7039])]))
    ref, sabs = og.gemm_w4a4(host(xq.codes).reshape(M, K // 2)[rows], host(xq.scales).reshape(M, K // 16)[rows],
                             float(host(xq.tensor_scale)[0]), host(wq.codes), host(wq.scales),
                             float(host(wq.tensor_scale)[0]))
    check(y[rows], ref, sabs, K)


def test_rht16_bit_exact(nv):
    """The transform against the oracle's butterflies, fp32 and bf16 inputs, bit for bit."""
    from nvfp4_block_quantization_gb300 import workloads as W
    from oracle import gemm as og

    rng = np.random.default_rng(21)
    x = (rng.standard_normal((37, 80)) * 3).astype(np.float32)
    got = host(nv.rht16(torch.from_numpy(x).cuda(), 0xB16B))
    assert np.array_equal(got.view(np.uint32), og.rht16(x, 0xB16B).view(np.uint32))
    xb = W.to_bf16_bits(W.activations(T=64, D=3072))
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    got = host(nv.rht16(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda(), 0x0F0F))
    assert np.array_equal(got.view(np.uint32), og.rht16(xf, 0x0F0F).view(np.uint32))


def test_w4a4_with_rht(nv):
    """Both operands transformed with the same signs, then quantized (fp32 inputs) and multiplied:
    within the bound of the oracle's product of the transformed, quantized operands."""
    from oracle import gemm as og

    rng = np.random.default_rng(13)
    M, N, K = 256, 512, 1024
    X = rng.standard_normal((M, K)).astype(np.float32)
    Wm = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Wm.flat[rng.choice(Wm.size, Wm.size // 1000, replace=False)] *= 30.0
    signs = int(rng.integers(0, 1 << 16))
    xr = nv.rht16(bf16_dev(X), signs)
    wr = nv.rht16(bf16_dev(Wm), signs)
    xq = nv.kv_smooth_quant(xr.view(M, 1, K), False)
    wq = nv.weight_quant_2d(wr)
    torch.cuda.synchronize()
    y = run_gemm(nv, xq, wq, M, N, K)
    ref, sabs = og.gemm_w4a4(host(xq.codes).reshape(M, K // 2), host(xq.scales).reshape(M, K // 16),
                             float(host(xq.tensor_scale)[0]), host(wq.codes), host(wq.scales),
                             float(host(wq.tensor_scale)[0]))
    check(y, ref, sabs, K)


def unswizzle(buf: np.ndarray, rows: int, KB: int) -> np.ndarray:
    """Block scales [rows][KB] read back out of the tensor-core layout."""
    kbt = (KB + 3) // 4
    r = np.arange(rows)[:, None]
    kb = np.arange(KB)[None, :]
    off = ((r // 128) * kbt + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    return buf[off]


@pytest.mark.parametrize("rht", [None, 0x9C3A], ids=["plain", "rht"])
@pytest.mark.parametrize("shape", [(200, 80), (7040, 3072)], ids=["200x80", "7040x3072"])
def test_act_quant_mma_equals_composition(nv, rht, shape):
    """The fused activation quantizer gives the separate calls' bits: codes, the whole scale
    buffer (padding included), tensor scale, status."""
    from nvfp4_block_quantization_gb300 import workloads as W

    M, K = shape
    X = W.activations(T=M, D=K, seed=5300 + K)
    X[:, ::97] *= 20.0  # outlier channels
    xb = bf16_dev(X)
    fused = nv.act_quant_mma(xb, rht)
    src = nv.rht16(xb, rht) if rht is not None else xb
    q = nv.kv_smooth_quant(src.view(M, 1, K), False)
    sm = nv.mma_scales(q.scales.view(M, K // 16), K)
    torch.cuda.synchronize()
    assert int(host(fused.status)[0]) == 0 and int(host(q.status)[0]) == 0
    assert torch.equal(fused.codes, q.codes.view(M, K // 2))
    n = nv._lib.nvfp4_mma_scales_bytes(M, K)
    assert torch.equal(fused.scales_mma[:n], sm[:n])
    assert torch.equal(fused.tensor_scale.view(torch.int32), q.tensor_scale.view(torch.int32))


@pytest.mark.parametrize("rht", [None, 0x2F51], ids=["plain", "rht"])
def test_act_quant_mma_matches_oracle(nv, oracle, rht):
    """Against the oracle's composition: (transform,) 1-D quantization, bit for bit."""
    from nvfp4_block_quantization_gb300 import workloads as W
    from oracle import gemm as og

    M, K = 150, 208
    X = W.activations(T=M, D=K, seed=5400)
    X[:, 5] *= 40.0
    bits = W.to_bf16_bits(X)
    fused = nv.act_quant_mma(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda(), rht)
    torch.cuda.synchronize()
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    src = og.rht16(xf, rht) if rht is not None else bits
    ref = oracle.kv_smooth_quant(src.reshape(M, 1, K), smooth=False)
    assert np.array_equal(host(fused.codes), ref["codes"].reshape(M, K // 2))
    assert np.array_equal(unswizzle(host(fused.scales_mma), M, K // 16), ref["scales"].reshape(M, K // 16))
    assert np.float32(host(fused.tensor_scale)[0]).view(np.uint32) == np.float32(ref["g"]).view(np.uint32)
