"""Pins of the oracle's head weights (w = w_scale * hidden @ w_proj^T from bf16 inputs):
bf16 decoding against known bit patterns, exact one-hot selections, zero, linearity and
permutation invariance on integer-valued inputs, and the error bound on same-sign terms."""
import numpy as np

import oracle


def bits(values):
    """float32 values that are exact bf16 -> their bf16 bit patterns."""
    v = np.asarray(values, np.float32)
    b = v.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "not exact bf16"
    return (b >> 16).astype(np.uint16)


def trunc_bits(values):
    """bf16 bit patterns of float32 values, truncated (any bf16 will do here)."""
    return (np.asarray(values, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_bf16_values_of_known_patterns():
    pats = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x0080, 0x3E80], np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 3.3895313892515355e38, 2.0 ** -133, 2.0 ** -126, 0.25]
    got = oracle.bf16_values(pats)
    assert list(got) == want
    assert np.signbit(got[3])


def test_one_hot_rows_select_a_column():
    rng = np.random.default_rng(0)
    H, D = 64, 256
    w = bits(rng.integers(-64, 64, size=(H, D)).astype(np.float32) / 8)
    hidden = np.zeros((5, D), np.uint16)
    cols = [0, 7, 128, 200, 255]
    for t, d in enumerate(cols):
        hidden[t, d] = 0x3F80  # 1.0
    got, bound = oracle.head_weights(hidden, w, 0.5)
    for t, d in enumerate(cols):
        assert np.array_equal(got[t], 0.5 * oracle.bf16_values(w)[:, d])
        assert np.array_equal(bound[t], np.abs(got[t]))


def test_zero_input_and_zero_scale():
    rng = np.random.default_rng(1)
    w = trunc_bits(rng.standard_normal((64, 512)))
    h = trunc_bits(rng.standard_normal((3, 512)))
    z, zb = oracle.head_weights(np.zeros((3, 512), np.uint16), w, 1.0)
    assert np.all(z == 0) and np.all(zb == 0)
    s, sb = oracle.head_weights(h, w, 0.0)
    assert np.all(s == 0) and np.all(sb == 0)


def test_linearity_and_permutation_on_integers():
    rng = np.random.default_rng(2)
    H, D = 8, 512
    x = rng.integers(-8, 9, size=(1, D)).astype(np.float32)
    y = rng.integers(-8, 9, size=(1, D)).astype(np.float32)
    w = rng.integers(-8, 9, size=(H, D)).astype(np.float32)
    wx, _ = oracle.head_weights(bits(x), bits(w), 1.0)
    wy, _ = oracle.head_weights(bits(y), bits(w), 1.0)
    wxy, _ = oracle.head_weights(bits(x + y), bits(w), 1.0)   # |x + y| <= 16: exact bf16
    w2x, _ = oracle.head_weights(bits(2 * x), bits(w), 1.0)
    assert np.array_equal(wxy, wx + wy)
    assert np.array_equal(w2x, 2 * wx)
    perm = rng.permutation(D)
    wp, _ = oracle.head_weights(bits(x[:, perm]), bits(w[:, perm]), 1.0)
    assert np.array_equal(wp, wx)
    # integer inputs: the value is the integer dot product
    assert np.array_equal(wx[0], (w.astype(np.int64) @ x[0].astype(np.int64)).astype(np.float64))


def test_bound_equals_magnitude_for_same_sign_terms():
    rng = np.random.default_rng(3)
    x = bits(rng.integers(1, 9, size=(2, 256)).astype(np.float32))
    w = bits(rng.integers(1, 9, size=(64, 256)).astype(np.float32))
    v, b = oracle.head_weights(x, w, -0.25)
    assert np.array_equal(b, -v) and np.all(v < 0)
