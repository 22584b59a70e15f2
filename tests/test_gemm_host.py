"""W4A4 NVFP4 GEMM without a GPU: the oracle reference against closed forms, and the
C entry points' argument checks (which return before any CUDA call)."""
import ctypes

import numpy as np
import pytest

from oracle import gemm as og


def test_reference_closed_form_scales():
    """Every element 1.0; activation block scales 1 (even blocks) and 0.5 (odd blocks) times
    (1 + m % 3); weight tile scales 2^(tile row % 4).  Each output is then a closed form."""
    M, N, K = 5, 64, 128
    KB = K // 16
    xc = np.full((M, K // 2), 0x22, np.uint8)       # E2M1 code 2 = 1.0 in both nibbles
    wc = np.full((N, K // 2), 0x22, np.uint8)
    one_two_three = [0x38, 0x40, 0x44]               # E4M3 1, 2, 3
    xs = np.array([[one_two_three[m % 3] if kb % 2 == 0 else 0x30 for kb in range(KB)] for m in range(M)], np.uint8)
    pow2 = [0x38, 0x40, 0x48, 0x50]                  # E4M3 1, 2, 4, 8
    ws = np.array([[pow2[t % 4]] * KB for t in range(N // 16)], np.uint8)
    y, s = og.gemm_w4a4(xc, xs, 0.25, wc, ws, 3.0)
    for m in range(M):
        for n in range(N):
            want = 0.75 * 16 * (2 ** ((n // 16) % 4)) * (KB // 2) * ((1 + m % 3) + 0.5)
            assert y[m, n] == want and s[m, n] == want


def test_reference_nibble_order_and_sign():
    """Byte j holds element 2j in its low nibble: X bytes 0x42 (1, 2), W bytes 0x0A (-1, 0)
    pair 1 with -1 and 2 with 0, so each byte contributes -1 (a swap in one operand would give 0
    or -2)."""
    K = 64
    xc = np.full((1, K // 2), 0x42, np.uint8)
    wc = np.full((16, K // 2), 0x0A, np.uint8)
    xs = np.full((1, K // 16), 0x38, np.uint8)
    ws = np.full((1, K // 16), 0x38, np.uint8)
    y, s = og.gemm_w4a4(xc, xs, 1.0, wc, ws, 1.0)
    assert np.all(y == -K / 2) and np.all(s == K / 2)


def test_reference_one_hot_rows_read_out_w():
    """X row m is 1.0 at k = m and 0 elsewhere, all scales 1: Y[m, n] is W's element (n, m).
    W's elements are all different along k and n, so a transposed operand, a swapped index
    or a wrong nibble order moves values.  E2M1 codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6;
    bit 3 is the sign."""
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    M, N, K = 32, 32, 32
    wcode = np.array([[(5 * n + 3 * k + n // 7) % 16 for k in range(K)] for n in range(N)], np.uint8)
    wc = (wcode[:, 0::2] | (wcode[:, 1::2] << 4)).astype(np.uint8)
    xcode = np.zeros((M, K), np.uint8)
    xcode[np.arange(M), np.arange(M)] = 2              # 1.0
    xc = (xcode[:, 0::2] | (xcode[:, 1::2] << 4)).astype(np.uint8)
    xs = np.full((M, K // 16), 0x38, np.uint8)
    ws = np.full((N // 16, K // 16), 0x38, np.uint8)
    y, s = og.gemm_w4a4(xc, xs, 1.0, wc, ws, 1.0)
    for m in range(M):
        for n in range(N):
            assert y[m, n] == e2m1[wcode[n, m]] and s[m, n] == abs(e2m1[wcode[n, m]])


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_quantization_gb300 import _lib
    from nvfp4_block_quantization_gb300.build import build

    build()
    return _lib


def test_mma_scale_bytes(lib):
    assert lib.nvfp4_mma_scales_bytes(200, 512) == 256 * 32
    assert lib.nvfp4_mma_scales_bytes(128, 64) == 128 * 4
    assert lib.nvfp4_mma_scales_bytes(1, 16) == 128 * 4
    assert lib.nvfp4_mma_scales_bytes(7040, 3072) == 7040 * 192
    assert lib.nvfp4_mma_scales_bytes(8, 24) == 0


def test_gemm_argument_errors(lib):
    p = ctypes.c_void_p()
    for M, N, K in ((0, 64, 64), (8, 24, 64), (8, 64, 48), (8, 64, 16), (1 << 31, 64, 64)):
        assert lib.nvfp4_gemm_plan_create(M, N, K, p) == lib.NVFP4_ESHAPE
        assert not p.value
    assert lib.load().nvfp4_gemm_plan_create(8, 64, 64, None) == lib.NVFP4_EINVAL
    g = 1 << 20
    assert lib.nvfp4_gemm_w4a4(None, g, g, g, g, g, g, g, g, 1 << 26, None) == lib.NVFP4_EINVAL
    assert lib.nvfp4_scales_to_mma(g, 8, 24, g, None) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_w2d_scales_to_mma(g, 24, 64, g, None) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_scales_to_mma(None, 8, 64, g, None) == lib.NVFP4_EINVAL


def test_rht16_unit_vectors_give_hadamard_rows():
    """The transform of unit vector e_i is row i of the Sylvester Hadamard matrix over 4,
    (-1)^popcount(i & j) / 4, negated when sign bit i is set."""
    E = np.eye(16, dtype=np.float32)
    H = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(16)] for i in range(16)]) / 4
    assert np.array_equal(og.rht16(E, 0), H.astype(np.float32))
    signs = 0b1010000000010011
    D = np.array([-1.0 if (signs >> i) & 1 else 1.0 for i in range(16)])
    assert np.array_equal(og.rht16(E, signs), (D[:, None] * H).astype(np.float32))


def test_rht16_is_orthogonal():
    """R = D H / 4 has R R^T = I: on small integers (every sum exact) the transform of the
    transform, with the signs applied after the butterflies, returns the input; and
    (X R)(W R)^T = X W^T exactly."""
    rng = np.random.default_rng(2)
    X = rng.integers(-8, 9, size=(6, 64)).astype(np.float32)
    Wm = rng.integers(-8, 9, size=(5, 64)).astype(np.float32)
    s = 0x5A3C
    Y = og.rht16(X, s)
    back = og.rht16(Y, 0)  # (x D H / 4) H / 4 = x D: undo D by the signs
    D = np.tile(np.array([-1.0 if (s >> i) & 1 else 1.0 for i in range(16)], np.float32), 4)
    assert np.array_equal(back * D, X)
    assert np.array_equal(Y.astype(np.float64) @ og.rht16(Wm, s).astype(np.float64).T,
                          X.astype(np.float64) @ Wm.astype(np.float64).T)


def test_rht16_argument_errors(lib):
    g = 1 << 20
    assert lib.nvfp4_rht16(g, 0, 4, 24, 0, g, None) == lib.NVFP4_ESHAPE
    assert lib.nvfp4_rht16(g, 0, 4, 32, 1 << 16, g, None) == lib.NVFP4_EINVAL
    assert lib.nvfp4_rht16(g, 2, 4, 32, 0, g, None) == lib.NVFP4_EINVAL
    assert lib.nvfp4_rht16(g + 16, 0, 4, 32, 0, g, None) == lib.NVFP4_EALIGN
    assert lib.nvfp4_rht16(None, 0, 4, 32, 0, g, None) == lib.NVFP4_EINVAL
    assert lib.nvfp4_rht16(None, 0, 0, 32, 0, None, None) == lib.NVFP4_OK


def test_act_quant_argument_errors(lib):
    """Checks that return before any CUDA call (the workspace check needs the device's SM count)."""
    g = 1 << 20
    L = lib.load()
    q = lambda x=g, M=64, K=128, rht=0, signs=0, codes=g, sf=g, ts=g: L.nvfp4_act_quant_mma(
        x, M, K, rht, signs, codes, sf, ts, None, g, 1 << 20, None)
    assert q(M=0) == lib.NVFP4_ESHAPE and q(K=24) == lib.NVFP4_ESHAPE and q(K=0) == lib.NVFP4_ESHAPE
    assert q(rht=2) == lib.NVFP4_EINVAL and q(signs=1 << 16) == lib.NVFP4_EINVAL
    assert q(x=None) == lib.NVFP4_EINVAL and q(ts=None) == lib.NVFP4_EINVAL
    assert q(x=g + 16) == lib.NVFP4_EALIGN and q(codes=g + 8) == lib.NVFP4_EALIGN and q(sf=g + 4) == lib.NVFP4_EALIGN


def test_bench_byte_accounting():
    """The bench's algorithmic bytes per element: 2 in + 0.5 codes + 1/16 scales (1-D blocks),
    0.5 + 1/16 in + 2 out (cache read), 2 + 0.5 + 1/256 (16x16 weight tiles)."""
    import importlib.util
    import os

    spec = importlib.util.spec_from_file_location(
        "bench_mod", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert b.QUANT_BYTES_PER_ELEM == 2.5625
    assert b.DEQUANT_BYTES_PER_ELEM == 2.5625
    assert b.W2D_BYTES_PER_ELEM == 2 + 0.5 + 1 / 256
    assert b.FP4_OVER_BF16 == 6.0
