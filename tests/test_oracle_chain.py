"""Pins of the oracle's row transforms (RMSNorm, RoPE, Hadamard) and of the whole
K/Q chains against closed forms, explicit matrices and float64 re-derivations."""
import numpy as np
import pytest

import oracle
from sparse_attention_fp4_gb300 import workloads as wl

F32_EPS = 2.0 ** -24


def sylvester(n):
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def test_hadamard_matrix_is_orthogonal_and_matches_butterfly():
    H = sylvester(128)
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    inv = np.float32(np.frombuffer(np.uint32(0x3DB504F3).tobytes(), np.float32)[0])
    assert abs(float(inv) - 128 ** -0.5) < 2 ** -27
    for i in range(128):
        e = np.zeros(128, np.float32)
        e[i] = 1.0
        # a unit vector goes through the butterflies without rounding: column i of H, times the scale
        assert np.array_equal(oracle.hadamard128(e), (H[:, i] * inv).astype(np.float32))


def test_hadamard_random_against_float64_and_norm():
    H = sylvester(128) / np.sqrt(128.0)
    rng = np.random.default_rng(0)
    for _ in range(200):
        x = (rng.standard_normal(128) * np.exp(rng.uniform(-3, 3))).astype(np.float32)
        y = oracle.hadamard128(x).astype(np.float64)
        ref = H @ x.astype(np.float64)
        # 7 add stages + 1 scaling, each error <= 2^-24 of the running |sum| <= ||x||_1
        tol = 9 * F32_EPS * np.abs(x).astype(np.float64).sum() / np.sqrt(128.0) * 2
        assert np.max(np.abs(y - ref)) <= tol
        assert abs(np.linalg.norm(y) - np.linalg.norm(x.astype(np.float64))) <= 1e-5 * np.linalg.norm(x)


def test_rmsnorm_constant_row_closed_form():
    for c in [0.5, 1.0, 3.0, -2.25, 1e-3, 40.0]:
        for wv in [1.0, 0.75, -1.5]:
            x = np.full(128, c, np.float32)
            w = np.full(128, wv, np.float32)
            y = oracle.rmsnorm(x, w, 1e-6)
            ref = wv * c / np.sqrt(c * c + 1e-6)
            assert np.allclose(y, ref, rtol=4 * F32_EPS, atol=0)
    y = oracle.rmsnorm(np.zeros(128, np.float32), np.ones(128, np.float32), 1e-6)
    assert np.all(y == 0)


def test_rmsnorm_random_against_float64():
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = (rng.standard_normal(128) * np.exp(rng.uniform(-4, 4))).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
        y = oracle.rmsnorm(x, w, 1e-6).astype(np.float64)
        xd = x.astype(np.float64)
        ref = xd / np.sqrt(np.mean(xd * xd) + float(np.float32(1e-6))) * w
        assert np.allclose(y, ref, rtol=32 * F32_EPS, atol=0)


def test_rope_conventions_and_rotation(cos_sin):
    assert np.all(wl.bf16_bits_to_f32(cos_sin[0, :32]) == 1.0) and np.all(wl.bf16_bits_to_f32(cos_sin[0, 32:]) == 0.0)
    rng = np.random.default_rng(2)
    u = rng.standard_normal(128).astype(np.float32)
    assert np.array_equal(oracle.rope(u, cos_sin[0]), u)               # position 0 is the identity
    p = 12345
    c = wl.bf16_bits_to_f32(cos_sin[p, :32]).astype(np.float64)
    s = wl.bf16_bits_to_f32(cos_sin[p, 32:]).astype(np.float64)
    for i in [0, 7, 31]:
        e = np.zeros(128, np.float32)
        e[i] = 1.0
        r = oracle.rope(e, cos_sin[p])
        assert r[i] == c[i] and r[i + 32] == s[i] and np.count_nonzero(r) <= 2   # (a,b)=(1,0) -> (cos, sin)
        e = np.zeros(128, np.float32)
        e[i + 32] = 1.0
        r = oracle.rope(e, cos_sin[p])
        assert r[i] == -s[i] and r[i + 32] == c[i]                                # (0,1) -> (-sin, cos)
    r = oracle.rope(u, cos_sin[p]).astype(np.float64)
    ud = u.astype(np.float64)
    ref = ud.copy()
    ref[:32] = ud[:32] * c - ud[32:64] * s
    ref[32:64] = ud[32:64] * c + ud[:32] * s
    assert np.allclose(r, ref, rtol=0, atol=4 * F32_EPS * np.abs(ud).max() * 2)
    assert np.array_equal(r[64:], ud[64:])
    # the bf16 table: cos^2 + sin^2 = 1 to bf16 precision
    assert np.all(np.abs(c * c + s * s - 1) < 2 ** -6)
    ang = p * 10000.0 ** (-2.0 * np.arange(32) / 64)
    assert np.all(np.abs(c - np.cos(ang)) <= 2 ** -8) and np.all(np.abs(s - np.sin(ang)) <= 2 ** -8)


def test_k_and_q_chain_against_float64(cos_sin):
    H = sylvester(128) / np.sqrt(128.0)
    ks = wl.small_kstore(3, 64, 1)
    nw = wl.bf16_bits_to_f32(ks.norm_w).astype(np.float64)
    for n in range(64):
        x = wl.bf16_bits_to_f32(ks.k_rows[n]).astype(np.float64)
        p = int(ks.positions[n])
        y = x / np.sqrt(np.mean(x * x) + float(np.float32(ks.eps))) * nw
        c = wl.bf16_bits_to_f32(cos_sin[p, :32]).astype(np.float64)
        s = wl.bf16_bits_to_f32(cos_sin[p, 32:]).astype(np.float64)
        a, b = y[:32].copy(), y[32:64].copy()
        y[:32], y[32:64] = a * c - b * s, b * c + a * s
        z = H @ y
        got = oracle.k_chain(ks.k_rows[n], p, ks.norm_w, ks.eps, cos_sin).astype(np.float64)
        assert np.max(np.abs(got - z)) <= 1e-5 * np.abs(z).max()
        q = ks.k_rows[n]
        xq = wl.bf16_bits_to_f32(q).astype(np.float64)
        a, b = xq[:32].copy(), xq[32:64].copy()
        xq[:32], xq[32:64] = a * c - b * s, b * c + a * s
        zq = H @ xq
        gotq = oracle.q_chain(q, p, cos_sin).astype(np.float64)
        assert np.max(np.abs(gotq - zq)) <= 1e-5 * np.abs(zq).max()


def test_quant_q_layout(cos_sin):
    rng = np.random.default_rng(4)
    T, Hh = 3, 64
    q = wl.f32_to_bf16_bits(rng.standard_normal((T, Hh, 128)).astype(np.float32))
    pos = np.array([0, 77, 131071], np.int32)
    qp, qs, st = oracle.quant_q(q, pos, cos_sin)
    assert st == 0 and qp.shape == (T, 4, Hh, 16) and qs.shape == (T, 4, Hh)
    for t in range(T):
        for h in [0, 5, 63]:
            z = oracle.q_chain(q[t, h], pos[t], cos_sin)
            pk, sc = oracle.fp4_encode_rows(z)
            assert np.array_equal(qp[t, :, h, :], pk[0]) and np.array_equal(qs[t, :, h], sc[0])
    _, _, st = oracle.quant_q(q, np.array([0, -1, 5], np.int32), cos_sin)
    assert st != 0
