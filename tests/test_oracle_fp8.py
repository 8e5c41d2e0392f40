"""Pins of the oracle's FP8 comparison path (132 B/token pages, FP8 query pack, FP8 logits).
The strongest: operands whose FP8 encoding dequantises to exactly the values of an FP4 cache
and FP4 query pack (e2m1 values times powers of two are e4m3 values too) must give
bit-identical logits to the FP4 oracle, which its own pins fix independently."""
import numpy as np

import oracle
from sparse_attention_fp4_gb300 import workloads as wl

CS = None


def cos_sin():
    global CS
    if CS is None:
        CS = wl.rope_cos_sin_table()
    return CS


def test_query_pack_layout_extreme_and_rounding_bound():
    b = wl.small_batch(1, [100], rows_per_seq=3, topk=8)
    q8, s8, st = oracle.quant_q_fp8(b.q, b.q_positions, cos_sin())
    assert st == 0 and q8.shape == (3, 8, 64, 16) and s8.shape == (3, 64)
    for t in range(3):
        for h in (0, 17, 63):
            z = oracle.q_chain(b.q[t, h], int(b.q_positions[t]), cos_sin()).astype(np.float64)
            sc = float(s8[t, h])
            assert sc == float(np.float32(np.float32(np.abs(z).max()) / np.float32(448.0)))
            codes = np.array([q8[t, i // 16, h, i % 16] for i in range(128)])
            vals = np.array([oracle.e4m3_value(int(c)) for c in codes])
            assert np.array_equal(oracle.dequant_q_fp8(q8, s8, t, h), vals * sc)  # layout [t][c][h][16]
            top = int(np.argmax(np.abs(z)))
            assert codes[top] & 0x7F == 0x7E  # the largest magnitude encodes to 448
            # round to nearest: within half a spacing of the e4m3 grid around z/s (2^-10 below 2^-6)
            x = np.abs(z / sc)
            e = np.floor(np.log2(np.maximum(x, 2.0 ** -6)))
            half = 2.0 ** (e - 4)
            assert np.all(np.abs(vals - z / sc) <= half * (1 + 1e-9) + 1e-300)


def test_zero_query_row():
    q = np.zeros((1, 64, 128), np.uint16)
    q8, s8, st = oracle.quant_q_fp8(q, np.zeros(1, np.int32), cos_sin())
    assert st == 0 and np.all(q8 == 0) and np.all(s8 == 1.0)


def test_k_token_dequant_matches_the_store():
    ks = wl.small_kstore(2, 40, 4)
    pages, st = oracle.store_k_fp8(ks, cos_sin())
    assert st == 0
    for n in (0, 7, 39):
        slot = int(ks.slots[n])
        p, j = slot // 64, slot % 64
        base = pages[p]
        sc = np.frombuffer(base[8192 + 4 * j:8192 + 4 * j + 4].tobytes(), np.float32)[0]
        want = np.array([oracle.e4m3_value(int(c)) for c in base[j * 128:(j + 1) * 128]]) * float(sc)
        assert np.array_equal(oracle.dequant_k_fp8_token(pages, p, j), want)


def fp8_twin_of_fp4(payload, scale, q_payload, q_scale):
    """FP8 pages and FP8 query pack whose dequantised values equal the FP4 ones exactly: per
    token (or row and head) the fp32 scale is 2^(smallest block exponent) and each value is
    re-encoded in e4m3 relative to it (e2m1 values times small powers of two are e4m3 values)."""
    P = payload.shape[0]
    pages = np.zeros((P, 64 * 132), np.uint8)
    for p in range(P):
        for j in range(64):
            v = oracle.dequant_k_token(payload, scale, p, j)
            e = int(scale[p, :, j].min()) - 127
            sc = np.float32(2.0 ** e)
            codes = [oracle.e4m3_codes(np.array([x / float(sc)], np.float32))[0] for x in v]
            back = np.array([oracle.e4m3_value(int(c)) for c in codes]) * float(sc)
            assert np.array_equal(back, v), "not representable"
            pages[p, j * 128:(j + 1) * 128] = codes
            pages[p, 8192 + 4 * j:8192 + 4 * j + 4] = np.frombuffer(sc.tobytes(), np.uint8)
    T, _, H, _ = q_payload.shape
    q8 = np.zeros((T, 8, H, 16), np.uint8)
    s8 = np.zeros((T, H), np.float32)
    for t in range(T):
        for h in range(H):
            v = oracle.dequant_q(q_payload, q_scale, t, h)
            e = int(q_scale[t, :, h].min()) - 127
            s8[t, h] = np.float32(2.0 ** e)
            for i, x in enumerate(v):
                q8[t, i // 16, h, i % 16] = oracle.e4m3_codes(np.array([x / float(s8[t, h])], np.float32))[0]
    return pages, q8, s8


def test_fp8_logits_equal_fp4_logits_on_shared_values():
    b = wl.small_batch(4, [130, 64, 1], rows_per_seq=2, topk=8)
    payload, scale, st = oracle.store_k(b.kstore, cos_sin())
    assert st == 0
    qp, qs, st = oracle.quant_q(b.q, b.q_positions, cos_sin())
    assert st == 0
    # keep every block exponent of a token within e4m3's reach of its smallest one
    assert int((scale.max(axis=1).astype(int) - scale.min(axis=1).astype(int)).max()) <= 6
    pages, q8, s8 = fp8_twin_of_fp4(payload, scale, qp, qs)
    lg4, bd4, st4 = oracle.logits(qp, qs, b.w, payload, scale, b.page_table, b.row_seq, b.context_lens)
    lg8, bd8, st8 = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens)
    assert st4 == 0 and st8 == 0
    assert np.array_equal(np.isnan(lg4), np.isnan(lg8))
    ok = ~np.isnan(lg4)
    assert np.array_equal(lg4[ok], lg8[ok]) and np.array_equal(bd4[ok], bd8[ok])


def test_fp8_logits_masking_and_bad_pages():
    b = wl.small_batch(5, [70, 0], rows_per_seq=1, topk=8)
    pages, st = oracle.store_k_fp8(b.kstore, cos_sin())
    q8, s8, _ = oracle.quant_q_fp8(b.q, b.q_positions, cos_sin())
    lg, bd, st = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens)
    assert st == 0
    assert np.all(~np.isnan(lg[0, :70])) and np.all(np.isnan(lg[1]))
    bad = b.page_table.copy()
    bad[0, 1] = pages.shape[0] + 5
    lg, _, st = oracle.logits_fp8(q8, s8, b.w, pages, bad, b.row_seq, b.context_lens)
    assert st == 5 and np.all(np.isnan(lg[0, 64:70])) and np.all(~np.isnan(lg[0, :64]))
