"""Pins of the attention reference (``oracle/attention.py``) without a GPU.

- Its fp32 dequant, rounded to bf16, is the C oracle's cache read (``kv_dequant``), bit
  for bit: two independent statements of the same formula.
- Closed forms of softmax attention: identical keys give the plain mean of V; one key
  far ahead of the others gives that token's V; adding a constant to every score
  changes nothing; two keys with score gap ln 3 / scale weigh 1/4 and 3/4 (also the bound's B).
"""
import numpy as np

from oracle import attention as oa


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """torch's round-to-nearest-even cast to bf16, as bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_dequant_matches_the_c_oracle(oracle):
    rng = np.random.default_rng(4)
    T, H, D = 40, 3, 32
    x = (rng.standard_normal((T, H, D)) * 2 + rng.standard_normal((1, H, D)) * 5).astype(np.float32)
    q = oracle.kv_smooth_quant(x, smooth=True)
    g = np.full(T, q["g"], np.float32)
    mean = np.broadcast_to(q["mean"], (T, H, D))
    v32 = oa.dequant_fp32(q["codes"], q["scales"], g, mean)
    ref = oracle.kv_dequant(q["codes"], q["scales"], q["g"], mean=q["mean"])
    assert np.array_equal(bf16_rne(v32), ref)
    v32n = oa.dequant_fp32(q["codes"], q["scales"], g)
    assert np.array_equal(bf16_rne(v32n), oracle.kv_dequant(q["codes"], q["scales"], q["g"]))


def test_identical_keys_give_the_mean_of_v():
    rng = np.random.default_rng(5)
    T, H, D = 9, 2, 16
    k = np.broadcast_to(rng.standard_normal((1, H, D)), (T, H, D))
    v = rng.standard_normal((T, H, D))
    q = rng.standard_normal((3, H, D))
    out, _, _ = oa.attention_decode(q, k, v, 0.25)
    assert np.allclose(out, np.broadcast_to(v.mean(axis=0), out.shape), rtol=0, atol=1e-12)


def test_a_dominant_key_selects_its_value():
    rng = np.random.default_rng(6)
    T, H, D = 7, 1, 16
    q = np.ones((1, H, D))
    k = rng.standard_normal((T, H, D)) * 0.01
    k[4] = 10.0  # score 160 / 4 = 40 above the others: weight 1 - O(e^-38)
    v = rng.standard_normal((T, H, D))
    out, _, _ = oa.attention_decode(q, k, v, 0.25)
    assert np.allclose(out[0, 0], v[4, 0], rtol=0, atol=1e-12)


def test_scores_shifted_by_a_constant_change_nothing():
    """Adding the same vector u to every key adds q . u to every score of a query: the
    softmax, and so the output, do not change."""
    rng = np.random.default_rng(7)
    T, H, D = 11, 2, 16
    q = rng.standard_normal((2, H, D))
    k = rng.standard_normal((T, H, D))
    v = rng.standard_normal((T, H, D))
    base, _, _ = oa.attention_decode(q, k, v, 0.3)
    u = rng.standard_normal((1, H, D))
    out_u, _, _ = oa.attention_decode(q, k + u, v, 0.3)
    assert np.allclose(out_u, base, rtol=0, atol=1e-12)


def test_two_keys_weighted_by_the_scaled_score_gap():
    """Two keys whose scores differ by c, with scale * c = ln 3: the softmax weights are
    exactly 1/4 and 3/4.  This fixes the softmax scale (dropped, squared or inverted, the
    weights move).  A and Vmax follow their definitions by hand."""
    D = 16
    q = np.zeros((1, 2, D))
    q[0, 0, :] = 1.0
    q[0, 1, 3] = -2.0
    c = 8.0
    scale = np.log(3.0) / c
    k = np.zeros((2, 2, D))
    k[1, 0, :] = c / D                   # head 0: q . k1 = c
    k[1, 1, 3] = -c / 2                  # head 1: q . k1 = c
    v = np.zeros((2, 2, D))
    v[0, :, :] = 4.0
    v[1, :, :] = -8.0
    v[1, 1, 5] = 12.0
    out, A, Vmax = oa.attention_decode(q, k, v, scale)
    want = 0.25 * v[0] + 0.75 * v[1]
    assert np.allclose(out[0], want, rtol=0, atol=1e-12)
    assert np.allclose(A[0], [scale * c, scale * c], rtol=1e-15, atol=0)
    assert np.array_equal(Vmax, [8.0, 12.0])


def test_weighted_abs_of_two_keys():
    """attention_weighted_abs on the same two-key case: weights exactly 1/4 and 3/4, so
    out = v0 / 4 + 3 v1 / 4 and B = |v0| / 4 + 3 |v1| / 4 per channel (B bounds how far a
    relative error in every weight can move the output).  Values of both signs, so a
    missing absolute value changes B."""
    D = 16
    q = np.zeros((1, 1, D))
    q[0, 0, :] = 1.0
    c = 8.0
    scale = np.log(3.0) / c
    k = np.zeros((2, 1, D))
    k[1, 0, :] = c / D
    v = np.zeros((2, 1, D))
    v[0, 0, :] = np.arange(D) - 7.5
    v[1, 0, :] = 3.0 - 0.5 * np.arange(D)
    out, B = oa.attention_weighted_abs(q, k, v, scale)
    assert np.allclose(out[0, 0], 0.25 * v[0, 0] + 0.75 * v[1, 0], rtol=0, atol=1e-12)
    assert np.allclose(B[0, 0], 0.25 * np.abs(v[0, 0]) + 0.75 * np.abs(v[1, 0]), rtol=0, atol=1e-12)
