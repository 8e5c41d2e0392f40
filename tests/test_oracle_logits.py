"""Pins of the oracle's paged-MQA logits and top-k.

* an independent numpy decoder of the split cache and a dense float64 einsum
  (brute force on tiny inputs),
* closed forms built from hand-written cache bytes (ReLU, weights, masking),
* invariants the pages state: identical results across page layouts and batch
  compositions, padded rows at length 0 empty, selections ordered by position.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_fp4_gb300 import workloads as wl

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def np_decode(pk, sc):
    """[...,4,16] bytes + [...,4] scales -> [...,128] float64 (independent of the C oracle)."""
    lo = E2M1[pk & 15]
    hi = E2M1[pk >> 4]
    v = np.stack([lo, hi], axis=-1).reshape(pk.shape[:-1] + (32,))
    v = v * np.exp2(sc.astype(np.float64) - 127)[..., None]
    return v.reshape(pk.shape[:-2] + (128,))


def brute_logits(qp, qs, w, payload, scale, page_table, row_seq, lens):
    q = np_decode(qp.transpose(0, 2, 1, 3), qs.transpose(0, 2, 1))          # [T,H,128]
    k = np_decode(payload.transpose(0, 2, 1, 3), scale.transpose(0, 2, 1))  # [P,64,128]
    out = []
    for t in range(qp.shape[0]):
        L = int(lens[t])
        s = np.arange(L)
        kk = k[page_table[row_seq[t], s // 64], s % 64]                     # [L,128]
        dots = np.einsum("hd,sd->sh", q[t], kk)
        out.append((np.maximum(dots, 0) * w[t][None, :].astype(np.float64)).sum(1))
    return out


def brute_topk(lg, k):
    L = lg.shape[0]
    order = np.lexsort((np.arange(L), -lg))[:min(k, L)]
    return np.concatenate([np.sort(order), -np.ones(k - order.size, np.int64)]).astype(np.int32)


@pytest.mark.parametrize("seed,lens,rows_per_seq,topk", [
    (10, [1, 63, 64, 65, 130], 1, 8),
    (11, [200, 7], 3, 16),
    (12, [0, 90], 2, 4),
])
def test_logits_and_topk_brute_force(cos_sin, seed, lens, rows_per_seq, topk):
    b = wl.small_batch(seed, lens, rows_per_seq=rows_per_seq, topk=topk)
    r = oracle.run_indexer(b, cos_sin)
    ref = brute_logits(r["q_payload"], r["q_scale"], b.w, r["payload"], r["scale"], b.page_table,
                       b.row_seq, b.context_lens)
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        got = r["logits"][t]
        assert np.all(np.isnan(got[L:]))
        assert np.allclose(got[:L], ref[t], rtol=1e-12, atol=1e-12)
        assert np.all(r["bound"][t][:L] >= np.abs(ref[t]) - 1e-9)
        assert np.array_equal(r["topk"][t], brute_topk(ref[t], topk))


def _const_token_cache(n_pages, k_codes_byte, k_scale_byte):
    payload = np.full((n_pages, 4, 64, 16), k_codes_byte, np.uint8)
    scale = np.full((n_pages, 4, 64), k_scale_byte, np.uint8)
    return payload, scale


def test_logits_closed_forms():
    # every q and k element is 1.0 (code 2 in both nibbles), scales 2^0: each head's dot = 128
    H, T = 64, 1
    qp = np.full((T, 4, H, 16), 0x22, np.uint8)
    qs = np.full((T, 4, H), 127, np.uint8)
    payload, scale = _const_token_cache(2, 0x22, 127)
    pt = np.array([[1, 0]], np.int32)
    w = np.full((T, H), 1.0 / 64, np.float32)
    lg, bnd, st = oracle.logits(qp, qs, w, payload, scale, pt, [0], [100])
    assert st == 0 and np.all(lg[0, :100] == 128.0) and np.all(bnd[0, :100] == 128.0)
    # negated k (sign nibbles): every dot = -128 -> ReLU gives 0
    payload_n, _ = _const_token_cache(2, 0xAA, 127)
    lg, _, _ = oracle.logits(qp, qs, w, payload_n, scale, pt, [0], [100])
    assert np.all(lg[0, :100] == 0.0)
    # half the heads see +q, half -q; weights 1..64: only the positive half counts
    qp2 = qp.copy()
    qp2[:, :, 32:, :] = 0xAA
    w2 = np.arange(1, 65, dtype=np.float32)[None, :]
    lg, _, _ = oracle.logits(qp2, qs, w2, payload, scale, pt, [0], [5])
    assert np.all(lg[0, :5] == 128.0 * np.arange(1, 33).sum())
    # scales: q block scale 2^3 on block 2 only, k scale 2^-2 everywhere -> dot = (32*3 + 32*8) * 2^-2 * ... per head
    qs3 = qs.copy()
    qs3[:, 2, :] = 130
    _, scale_m = _const_token_cache(2, 0x22, 125)
    lg, _, _ = oracle.logits(qp, qs3, w, payload, scale_m, pt, [0], [3])
    assert np.all(lg[0, :3] == (96 * 0.25 + 32 * 8 * 0.25))
    # a negative weight on a positive head subtracts
    w4 = w.copy()
    w4[0, 0] = -2.0
    lg, _, _ = oracle.logits(qp, qs, w4, payload, scale, pt, [0], [1])
    assert lg[0, 0] == 128.0 * (63 / 64 - 2.0)


def test_masking_padding_and_topk_edges(cos_sin):
    b = wl.small_batch(20, [0, 5, 70], rows_per_seq=1, topk=16)
    r = oracle.run_indexer(b, cos_sin)
    assert np.all(r["topk"][0] == -1)                                   # a padded row at length 0 is empty
    assert np.array_equal(r["topk"][1], np.r_[np.arange(5), -np.ones(11)])  # L <= k keeps every token, ascending
    t2 = r["topk"][2]
    assert np.all(np.diff(t2) > 0) and t2.min() >= 0 and t2.max() < 70  # ascending positions
    # all-equal logits: ties resolve to the lowest positions
    assert np.array_equal(oracle.topk(np.zeros(50), 50, 8), np.arange(8))
    lg = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 0.5])
    assert np.array_equal(oracle.topk(lg, 6, 2), [1, 2])
    assert np.array_equal(oracle.topk(lg, 6, 4), [1, 2, 3, 4])


def test_page_layout_and_batch_invariance(cos_sin):
    b = wl.small_batch(30, [150, 64, 90], rows_per_seq=2, topk=12)
    r = oracle.run_indexer(b, cos_sin)
    # move every physical page to a new location
    rng = np.random.default_rng(0)
    P = b.num_pages
    perm = rng.permutation(P)
    payload2 = np.empty_like(r["payload"])
    scale2 = np.empty_like(r["scale"])
    payload2[perm] = r["payload"]
    scale2[perm] = r["scale"]
    pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    lg2, _, st = oracle.logits(r["q_payload"], r["q_scale"], b.w, payload2, scale2, pt2, b.row_seq,
                               b.context_lens)
    assert st == 0 and np.array_equal(lg2, r["logits"], equal_nan=True)
    # one row alone == the same row inside the batch
    t = 3
    lg1, _, _ = oracle.logits(r["q_payload"][t:t + 1], r["q_scale"][t:t + 1], b.w[t:t + 1], r["payload"],
                              r["scale"], b.page_table, b.row_seq[t:t + 1], b.context_lens[t:t + 1])
    L = int(b.context_lens[t])
    assert np.array_equal(lg1[0, :L], r["logits"][t, :L])


def test_bad_page_is_reported():
    qp = np.full((1, 4, 64, 16), 0x22, np.uint8)
    qs = np.full((1, 4, 64), 127, np.uint8)
    payload, scale = _const_token_cache(2, 0x22, 127)
    w = np.ones((1, 64), np.float32)
    _, _, st = oracle.logits(qp, qs, w, payload, scale, np.array([[0, 7]], np.int32), [0], [100])
    assert st == 5
