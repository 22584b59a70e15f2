"""The C oracle against the independent numpy statement (oracle/restated.py), bit for bit.

The two statements share no code: the C oracle rounds with the formats' defining
arithmetic (frexp/nearbyint on the scaled value) and sums the error with C's
fmaf, the numpy statement searches the formats' value tables for the nearest
value and emulates the fused multiply-add in binary64.  A slip in either (a
wrong tie rule, a transposed tile, a skipped element, a dropped term) shows as
a difference here.
"""
import os
import json

import numpy as np
import pytest

from oracle import restated as R

HERE = os.path.dirname(os.path.abspath(__file__))


def _same_kv(a, b, smooth):
    assert a["status"] == b["status"]
    assert np.float32(a["g"]).view(np.uint32) == np.float32(b["g"]).view(np.uint32)
    if smooth:
        assert np.array_equal(np.ravel(a["mean"]).view(np.uint32), np.ravel(b["mean"]).view(np.uint32))
    assert np.array_equal(a["scales"], b["scales"])
    assert np.array_equal(a["codes"], b["codes"])


def test_tiny_config_both_statements_agree(oracle):
    from nvfp4_block_quantization_gb300 import workloads as W

    K, V = W.tiny_kv(0)
    _same_kv(oracle.kv_smooth_quant(K, smooth=True), R.kv_smooth_quant(K, True), True)
    _same_kv(oracle.kv_smooth_quant(V, smooth=False), R.kv_smooth_quant(V, False), False)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_bf16_both_statements_agree(oracle, seed):
    from nvfp4_block_quantization_gb300 import workloads as W

    x = W.to_bf16_bits(W.random_kv(seed, 192, 3, 64, scale=float(seed)))
    for smooth in (True, False):
        _same_kv(oracle.kv_smooth_quant(x, smooth=smooth), R.kv_smooth_quant(x, smooth), smooth)


def test_chunk_slice_both_statements_agree(oracle):
    """The first 384 tokens of the chunk workload (outlier channels x16 included)."""
    from nvfp4_block_quantization_gb300 import workloads as W

    K = W.to_bf16_bits(W.chunk_k(2000))[:384]
    V = W.to_bf16_bits(W.chunk_v(2001))[:384]
    _same_kv(oracle.kv_smooth_quant(K, smooth=True), R.kv_smooth_quant(K, True), True)
    _same_kv(oracle.kv_smooth_quant(V, smooth=False), R.kv_smooth_quant(V, False), False)


def test_hand_worked_tensors_both_statements_agree(oracle):
    with open(os.path.join(HERE, "golden", "hand_blocks.json")) as f:
        fx = json.load(f)
    row = np.concatenate([np.asarray(b["values"], np.float32) for b in fx["blocks"]])
    x = row.reshape(1, 1, -1)
    _same_kv(oracle.kv_smooth_quant(x, smooth=False), R.kv_smooth_quant(x, False), False)
    t = np.zeros((1, 1, 32), np.float32)
    t[0, 0, 0], t[0, 0, 16] = 23.0, 17.25   # the E4M3 tie of candidate_scale_tie.json
    _same_kv(oracle.kv_smooth_quant(t, smooth=False), R.kv_smooth_quant(t, False), False)


def test_degenerate_tensors_both_statements_agree(oracle):
    z = np.zeros((4, 2, 32), np.float32)
    _same_kv(oracle.kv_smooth_quant(z, smooth=True), R.kv_smooth_quant(z, True), True)
    c = np.full((8, 1, 16), 3.0, np.float32)           # constant channels: smoothed to zero
    _same_kv(oracle.kv_smooth_quant(c, smooth=True), R.kv_smooth_quant(c, True), True)
    tiny = np.full((2, 1, 16), 1e-38, np.float32)       # subnormal scales, unusable candidates
    tiny[0, 0, 3] = -2e-38
    _same_kv(oracle.kv_smooth_quant(tiny, smooth=False), R.kv_smooth_quant(tiny, False), False)
    bad = np.ones((2, 1, 16), np.float32)
    bad[1, 0, 5] = np.inf
    a, b = oracle.kv_smooth_quant(bad, smooth=False), R.kv_smooth_quant(bad, False)
    assert a["status"] == b["status"] == oracle.NONFINITE
    assert np.array_equal(a["scales"], b["scales"]) and np.array_equal(a["codes"], b["codes"])


@pytest.mark.parametrize("seed,shape", [(0, (64, 128)), (1, (128, 256)), (2, (48, 80))])
def test_weights_2d_both_statements_agree(oracle, seed, shape):
    from nvfp4_block_quantization_gb300 import workloads as W

    w = W.to_bf16_bits(W.weight(seed, *shape))
    a, b = oracle.weight_quant_2d(w), R.weight_quant_2d(w)
    assert np.float32(a["g"]).view(np.uint32) == np.float32(b["g"]).view(np.uint32)
    assert np.array_equal(a["scales"], b["scales"])
    assert np.array_equal(a["codes"], b["codes"])


def test_restated_minifloats_match_the_c_encoders(oracle):
    rng = np.random.default_rng(3)
    x = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(R.e2m1_encode(x), oracle.e2m1_encode_array(x))
    assert np.array_equal(R.e4m3_encode(x), oracle.e4m3_encode_array(x))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 336.0, 448.0, 464.0, 2.0 ** -10], np.float32)
    assert np.array_equal(R.e2m1_encode(mids), oracle.e2m1_encode_array(mids))
    assert np.array_equal(R.e4m3_encode(mids), oracle.e4m3_encode_array(mids))


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_threaded_driver_equals_the_single_threaded_oracle(oracle, threads):
    """The multi-threaded driver used to time the baseline on all cores splits channels, elements
    and blocks among threads; its outputs must be the single-threaded statement's, bit for bit."""
    from nvfp4_block_quantization_gb300 import workloads as W

    K = W.to_bf16_bits(W.chunk_k(2000))[:200]
    V = W.to_bf16_bits(W.chunk_v(2001))[:200]
    for x, smooth in ((K, True), (V, False), (W.tiny_kv(0)[0], True)):
        a, b = oracle.kv_smooth_quant(x, smooth=smooth), oracle.kv_smooth_quant_threads(x, smooth, threads)
        assert a["status"] == b["status"]
        assert np.float32(a["g"]).view(np.uint32) == np.float32(b["g"]).view(np.uint32)
        if smooth:
            assert np.array_equal(a["mean"].view(np.uint32), b["mean"].view(np.uint32))
        assert np.array_equal(a["scales"], b["scales"]) and np.array_equal(a["codes"], b["codes"])
    bad = np.ones((3, 1, 16), np.float32)
    bad[2, 0, 7] = np.nan
    assert oracle.kv_smooth_quant_threads(bad, False, threads)["status"] == oracle.NONFINITE
