"""GPU whole-page access to the split cache against the oracle.  Dequantised pages
equal the oracle's binary64 values rounded to fp32; every value is an e2m1 code times a
power of two, so this is exact, with +-inf past the fp32 range and subnormals at the
smallest scales.  Export then import moves pages byte for byte.  Padding ids are skipped
and ids past the cache are reported, not faulted."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def random_cache(seed, num_pages):
    """Random bytes: every e2m1 code with both signs, and scale bytes 0..254."""
    rng = np.random.default_rng(seed)
    payload = rng.integers(0, 256, size=(num_pages, 4, 64, 16), dtype=np.uint8)
    scale = rng.integers(0, 255, size=(num_pages, 4, 64), dtype=np.uint8)
    return payload, scale


def fp4():
    from sparse_attention_fp4_gb300 import fp4idx
    return fp4idx


def test_dequant_pages_matches_oracle():
    f = fp4()
    payload, scale = random_cache(1, 37)
    scale[3] = 254        # 2^127: codes >= 2 overflow fp32
    scale[4, 0, :5] = 253
    scale[5] = 0          # 2^-127: subnormal results
    ids = np.array([5, -1, 3, 36, 0, 4, 3], np.int32)
    out = torch.full((len(ids), 64, 128), 7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f.dequant_pages(dev(payload), dev(scale), dev(ids), out, status=status)
    got = host(out)
    assert f.read_status(status) == 0
    for i, p in enumerate(ids):
        if p < 0:
            assert np.all(got[i] == 7.0), "padding entry written"
            continue
        for j in range(64):
            with np.errstate(over="ignore"):
                ref = oracle.dequant_k_token(payload, scale, int(p), j).astype(np.float32)
            assert np.array_equal(got[i, j], ref), (i, int(p), j)
    assert np.any(np.isinf(got[2]))  # page 3 at scale 254: |value| >= 2^128 is +-inf
    assert np.any((got[0] != 0) & (np.abs(got[0]) < np.finfo(np.float32).tiny))  # page 5: subnormals


def test_export_import_round_trip():
    f = fp4()
    src_p, src_s = random_cache(2, 50)
    dst_p, dst_s = random_cache(3, 40)
    ids = np.array([7, 49, -1, 0, 23, 12], np.int32)
    tgt = np.array([39, 0, -1, 17, 5, 30], np.int32)
    rows_p = torch.full((len(ids), 4096), 0xAB, dtype=torch.uint8, device="cuda")
    rows_s = torch.full((len(ids), 256), 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f.export_pages(dev(src_p), dev(src_s), dev(ids), rows_p, rows_s, status=status)
    rp, rs = host(rows_p), host(rows_s)
    for i, p in enumerate(ids):
        if p < 0:
            assert np.all(rp[i] == 0xAB) and np.all(rs[i] == 0xCD), "padding row written"
        else:
            assert np.array_equal(rp[i], src_p[p].reshape(-1)) and np.array_equal(rs[i], src_s[p].reshape(-1)), i
    cache_p, cache_s = dev(dst_p), dev(dst_s)
    f.import_pages(rows_p, rows_s, dev(tgt), cache_p, cache_s, status=status)
    exp_p, exp_s = dst_p.copy(), dst_s.copy()
    for i, t in enumerate(tgt):
        if t >= 0:
            exp_p[t], exp_s[t] = src_p[ids[i]], src_s[ids[i]]
    assert np.array_equal(host(cache_p), exp_p) and np.array_equal(host(cache_s), exp_s)
    assert f.read_status(status) == 0


def test_pages_past_the_cache_are_reported():
    f = fp4()
    payload, scale = random_cache(4, 10)
    ids = np.array([3, 10, 4, 2 ** 31 - 1], np.int32)
    rows_p = torch.zeros((4, 4096), dtype=torch.uint8, device="cuda")
    rows_s = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    f.export_pages(dev(payload), dev(scale), dev(ids), rows_p, rows_s, status=status)
    assert f.read_status(status) == 5  # FP4IDX_ERR_BAD_PAGE
    rp = host(rows_p)
    assert np.array_equal(rp[0], payload[3].reshape(-1)) and np.array_equal(rp[2], payload[4].reshape(-1))
    assert np.all(rp[1] == 0) and np.all(rp[3] == 0)
    out = torch.zeros((4, 64, 128), dtype=torch.float32, device="cuda")
    status.zero_()
    f.dequant_pages(dev(payload), dev(scale), dev(ids), out, status=status)
    assert f.read_status(status) == 5
    assert np.all(host(out)[1] == 0)
