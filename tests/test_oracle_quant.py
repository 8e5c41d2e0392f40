"""Pins of the oracle's quantisation steps against definitions that do not share its code.

e2m1 is checked against IEEE round-half-even on the format's quantum (numpy's
round), e4m3 against torch's float8_e4m3fn cast, UE8M0 against its closed-form
exponent, the packed layout against the byte counts the pages print.
"""
import json
import os

import numpy as np
import pytest

import oracle
from sparse_attention_fp4_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rne_e2m1_by_quantum(v):
    """Independent e2m1 RNE: round |v| to the format's quantum at its binade with
    half-even integer rounding, saturate at 6, return the code."""
    v = np.asarray(v, np.float64)
    m = np.abs(v)
    q = np.where(m < 2.0, 0.5, np.where(m < 4.0, 1.0, 2.0))
    r = np.minimum(np.round(m / q) * q, 6.0)
    code = np.searchsorted(GRID, r)
    assert np.all(GRID[code] == r)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def test_e2m1_all_codes_round_trip():
    for c in range(16):
        v = oracle.e2m1_value(c)
        if c == 8:
            assert v == 0.0
            assert oracle.e2m1_codes(np.array([-0.0], np.float32))[0] == 8
            continue
        assert oracle.e2m1_codes(np.array([v], np.float32))[0] == c
    assert [oracle.e2m1_value(c) for c in range(8)] == list(GRID)


def test_e2m1_midpoints_go_to_even_code():
    mids = (GRID[:-1] + GRID[1:]) / 2
    expect_code = [0, 2, 2, 4, 4, 6, 6]  # 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    got = oracle.e2m1_codes(mids.astype(np.float32))
    assert list(got) == expect_code
    got_neg = oracle.e2m1_codes((-mids).astype(np.float32))
    assert list(got_neg) == [c | 8 for c in expect_code]
    # one ulp either side of every midpoint
    up = np.nextafter(mids.astype(np.float32), np.float32(np.inf))
    dn = np.nextafter(mids.astype(np.float32), np.float32(-np.inf))
    assert list(oracle.e2m1_codes(up)) == list(range(1, 8))
    assert list(oracle.e2m1_codes(dn)) == list(range(0, 7))


def test_e2m1_dense_sweep_matches_quantum_rounding():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        np.linspace(-8, 8, 400_001, dtype=np.float32),
        rng.uniform(-7, 7, 200_000).astype(np.float32),
        np.array([0.0, -0.0, 6.0, -6.0, 1e30, -1e30, 1e-45, -1e-45], np.float32),
    ])
    assert np.array_equal(oracle.e2m1_codes(v), rne_e2m1_by_quantum(v))


def test_ue8m0_exponent_closed_form():
    for e in range(-120, 120, 7):
        a = np.float32(6.0 * 2.0 ** e)
        assert oracle.ue8m0_bytes([a])[0] == e + 127            # 6*2^e exactly fits
        a_up = np.nextafter(a, np.float32(np.inf))
        assert oracle.ue8m0_bytes([a_up])[0] == e + 128          # just above needs e+1
        a_half = np.float32(3.0 * 2.0 ** e)
        assert oracle.ue8m0_bytes([a_half])[0] == e + 126        # 3*2^e = 6*2^(e-1)
    assert oracle.ue8m0_bytes([0.0])[0] == 0
    assert oracle.ue8m0_bytes([1e-45])[0] == 0                   # clamp at 2^-127
    assert oracle.ue8m0_bytes([np.finfo(np.float32).max])[0] <= 254
    rng = np.random.default_rng(1)
    a = np.exp(rng.uniform(-60, 60, 100_000)).astype(np.float32)
    b = oracle.ue8m0_bytes(a).astype(np.int64)
    e = b - 127
    # smallest e with 6*2^e >= amax
    assert np.all(6.0 * np.exp2(e.astype(np.float64)) >= a.astype(np.float64))
    assert np.all(6.0 * np.exp2(e.astype(np.float64) - 1) < a.astype(np.float64))
    # against ceil(log2(amax/6)) away from the exact boundaries
    r = np.log2(a.astype(np.float64) / 6.0)
    far = np.abs(r - np.round(r)) > 1e-6
    assert np.array_equal(e[far], np.ceil(r[far]).astype(np.int64))


def test_e4m3_matches_torch_cast():
    torch = pytest.importorskip("torch")
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = np.array([oracle.e4m3_value(c) for c in codes], np.float32)
    got = oracle.e4m3_codes(vals)
    assert list(got) == codes
    assert oracle.e4m3_value(0x7E) == 448.0
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.uniform(-448, 448, 200_000), rng.normal(0, 1, 100_000),
                        rng.normal(0, 0.01, 100_000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_codes(v), ref)
    # saturation (torch's cast does not saturate, so this is the definition itself)
    assert list(oracle.e4m3_codes(np.array([449, 500, 1e9, -1e9], np.float32))) == [0x7E, 0x7E, 0x7E, 0xFE]


def test_fp4_encode_decode_error_bound_and_value_idempotence():
    rng = np.random.default_rng(3)
    z = (rng.standard_normal((2000, 128)) * np.exp(rng.uniform(-5, 5, (2000, 1)))).astype(np.float32)
    z[0] = 0.0
    z[1, :32] = 6.0
    pk, sc = oracle.fp4_encode_rows(z)
    zh = oracle.fp4_decode_rows(pk, sc)
    e = sc.astype(np.int64) - 127
    scale = np.exp2(np.repeat(e, 32, axis=1).astype(np.float64))
    v = np.abs(z.astype(np.float64)) / scale
    half_step = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    assert np.all(np.abs(zh - z) <= half_step * scale)
    assert np.all(v <= 6.0)                                         # the scale rule never saturates
    pk2, sc2 = oracle.fp4_encode_rows(zh.astype(np.float32))
    assert np.array_equal(oracle.fp4_decode_rows(pk2, sc2), zh)     # dequantised values are a fixed point


def test_packed_nibble_order_and_block_layout():
    z = np.zeros((1, 128), np.float32)
    z[0, 0] = 1.0     # block 0, byte 0, low nibble
    z[0, 1] = -6.0    # block 0, byte 0, high nibble
    z[0, 33] = 0.5    # block 1, byte 0, high nibble
    z[0, 127] = 3.0   # block 3, byte 15, high nibble
    pk, sc = oracle.fp4_encode_rows(z)
    assert sc[0, 0] == 127 and sc[0, 1] == 127 - 3 and sc[0, 3] == 127 - 1
    # block 0: amax 6 -> e = 0: 1.0 -> code 2, -6 -> code 15
    assert pk[0, 0, 0] == (2 | (15 << 4))
    # block 1: amax 0.5 -> e = -3: 0.5 * 8 = 4 -> code 6
    assert pk[0, 1, 0] == (6 << 4)
    # block 3: amax 3 -> e = -1: 3 * 2 = 6 -> code 7
    assert pk[0, 3, 15] == (7 << 4)


def test_split_cache_layout_and_sizes(cos_sin):
    with open(os.path.join(GOLDEN, "layout.json")) as f:
        g = json.load(f)
    assert g["fp4_payload_bytes_per_token"] + g["fp4_scale_bytes_per_token"] == g["fp4_bytes_per_token"] == 68
    assert 128 * 4 // 8 + 128 // 32 == g["fp4_bytes_per_token"]
    assert 128 + 4 == g["fp8_bytes_per_token"]
    assert int(np.prod(g["payload_shape_per_page"])) == 64 * g["fp4_payload_bytes_per_token"]
    assert int(np.prod(g["scale_shape_per_page"])) == 64 * g["fp4_scale_bytes_per_token"]
    assert oracle.FP8_PAGE_BYTES == 64 * g["fp8_bytes_per_token"]

    # one stored row touches exactly its 64 payload bytes and 4 scale bytes
    ks = wl.small_kstore(5, 1, 3)
    ks.slots[:] = 2 * 64 + 17
    payload, scale, st = oracle.store_k(ks, cos_sin)
    assert st == 0
    z = oracle.k_chain(ks.k_rows[0], ks.positions[0], ks.norm_w, ks.eps, cos_sin)
    pk, sc = oracle.fp4_encode_rows(z)
    expect_p = np.zeros_like(payload)
    expect_s = np.zeros_like(scale)
    expect_p[2, :, 17, :] = pk[0]
    expect_s[2, :, 17] = sc[0]
    assert np.array_equal(payload, expect_p) and np.array_equal(scale, expect_s)
    assert (payload != 0).sum() + (scale != 0).sum() <= g["fp4_bytes_per_token"]

    pages, st = oracle.store_k_fp8(ks, cos_sin)
    assert st == 0
    nz = np.nonzero(pages[2])[0]
    assert nz.min() >= 17 * 128 and (nz < 18 * 128).sum() + ((nz >= 8192 + 17 * 4) & (nz < 8192 + 18 * 4)).sum() == nz.size


def test_store_skips_padding_and_flags_bad_slots(cos_sin):
    ks = wl.small_kstore(6, 40, 2, pad_every=3)
    payload, scale, st = oracle.store_k(ks, cos_sin)
    assert st == 0
    written = set(int(s) for s in ks.slots if s >= 0)
    for page in range(2):
        for j in range(64):
            touched = payload[page, :, j].any() or scale[page, :, j].any()
            if page * 64 + j not in written:
                assert not touched
    ks.slots[5] = 2 * 64  # one past the cache
    _, _, st = oracle.store_k(ks, cos_sin)
    assert st == 5


def test_fp8_store_scale_rule(cos_sin):
    ks = wl.small_kstore(7, 64, 1)
    pages, st = oracle.store_k_fp8(ks, cos_sin)
    assert st == 0
    for n in range(64):
        z = oracle.k_chain(ks.k_rows[n], ks.positions[n], ks.norm_w, ks.eps, cos_sin).astype(np.float32)
        j = int(ks.slots[n]) % 64
        s = pages[0, 8192 + 4 * j: 8192 + 4 * j + 4].view(np.float32)[0]
        assert s == np.float32(np.abs(z).max()) / np.float32(448.0)
        codes = pages[0, j * 128:(j + 1) * 128]
        deq = np.array([oracle.e4m3_value(int(c)) for c in codes]) * float(s)
        # e4m3 has 3 mantissa bits: relative error <= 2^-4 for normals, plus the subnormal quantum
        assert np.all(np.abs(deq - z) <= np.abs(z) * 2.0 ** -4 + float(s) * 2.0 ** -10)
