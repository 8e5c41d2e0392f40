"""GPU parity: K store (FP4 split and FP8 fused layouts) and query packing must be
byte-identical to the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fx():
    from sparse_attention_fp4_gb300 import fp4idx
    cs = wl.rope_cos_sin_table()
    from tests.gpu_util import bf16
    return fp4idx, cs, bf16(cs)


def _gpu_store(fp4idx, cs_dev, ks, status=None):
    from tests.gpu_util import kstore_to_device
    d = kstore_to_device(ks)
    payload, scale = fp4idx.alloc_cache(ks.num_pages)
    fp4idx.store_k(d["k"], d["positions"], d["slots"], d["norm_w"], ks.eps, cs_dev, payload, scale, status=status)
    torch.cuda.synchronize()
    return payload.cpu().numpy(), scale.cpu().numpy()


def _assert_cache_equal(got_p, got_s, ref_p, ref_s):
    if not np.array_equal(got_s, ref_s):
        bad = np.argwhere(got_s != ref_s)
        raise AssertionError("scale mismatch at %d places, first %s: gpu %d oracle %d" % (
            len(bad), bad[0], got_s[tuple(bad[0])], ref_s[tuple(bad[0])]))
    if not np.array_equal(got_p, ref_p):
        bad = np.argwhere(got_p != ref_p)
        raise AssertionError("payload mismatch at %d places, first %s: gpu %#x oracle %#x" % (
            len(bad), bad[0], got_p[tuple(bad[0])], ref_p[tuple(bad[0])]))


def test_store_k_full_kstore_workload(fx):
    fp4idx, cs, cs_dev = fx
    ks = wl.kstore_65536()
    got_p, got_s = _gpu_store(fp4idx, cs_dev, ks)
    ref_p, ref_s, st = oracle.store_k(ks, cs)
    assert st == 0
    _assert_cache_equal(got_p, got_s, ref_p, ref_s)


# 40,003 rows: more rows than one pass of the resident CTAs covers, so warps loop, and
# the last pass ends in a partial warp
@pytest.mark.parametrize("n,pages,pad", [(1, 1, 0), (15, 1, 0), (17, 2, 3), (1000, 20, 7), (4097, 70, 0),
                                         (40003, 700, 11)])
def test_store_k_small_ragged(fx, n, pages, pad):
    fp4idx, cs, cs_dev = fx
    ks = wl.small_kstore(100 + n, n, pages, pad_every=pad)
    got_p, got_s = _gpu_store(fp4idx, cs_dev, ks)
    ref_p, ref_s, _ = oracle.store_k(ks, cs)
    _assert_cache_equal(got_p, got_s, ref_p, ref_s)


def test_store_k_edge_values(fx):
    """Zero rows, constant rows, huge and tiny magnitudes, negative norm weights:
    exercises signed zeros, clamped exponents and subnormal intermediates."""
    fp4idx, cs, cs_dev = fx
    ks = wl.small_kstore(7, 64, 1)
    rows = wl.bf16_bits_to_f32(ks.k_rows).copy()
    rows[0] = 0.0
    rows[1] = 1.0
    rows[2] = -3.0e38
    rows[3] = 1e-38
    rows[4, :64] = 0.0
    rows[5] = np.where(np.arange(128) % 2 == 0, 1e30, -1e-30)
    rows[6] = 2.0 ** -133
    ks.k_rows = wl.f32_to_bf16_bits(rows)
    nw = wl.bf16_bits_to_f32(ks.norm_w).copy()
    nw[::3] *= -1
    ks.norm_w = wl.f32_to_bf16_bits(nw)
    ks.positions[:8] = [0, 1, 131071, 65536, 2, 3, 4, 5]
    got_p, got_s = _gpu_store(fp4idx, cs_dev, ks)
    ref_p, ref_s, _ = oracle.store_k(ks, cs)
    _assert_cache_equal(got_p, got_s, ref_p, ref_s)


def test_store_k_reports_bad_slot_and_position(fx):
    fp4idx, cs, cs_dev = fx
    ks = wl.small_kstore(8, 100, 2)
    ks.slots[10] = 2 * 64 + 5          # past the cache
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got_p, got_s = _gpu_store(fp4idx, cs_dev, ks, status)
    assert fp4idx.read_status(status) == 5
    ref_p, ref_s, st = oracle.store_k(ks, cs)
    assert st == 5
    _assert_cache_equal(got_p, got_s, ref_p, ref_s)  # every valid row still lands
    ks2 = wl.small_kstore(9, 10, 1)
    ks2.positions[3] = cs.shape[0]
    status.zero_()
    _gpu_store(fp4idx, cs_dev, ks2, status)
    assert fp4idx.read_status(status) == 7


@pytest.mark.parametrize("n,pages,pad", [(17, 2, 3), (40003, 700, 11), (65536, 2048, 0)],
                         ids=["17", "40003", "kstore_65536"])
def test_store_k_fp8_against_oracle(fx, n, pages, pad):
    fp4idx, cs, cs_dev = fx
    from tests.gpu_util import kstore_to_device
    ks = wl.kstore_65536() if n == 65536 else wl.small_kstore(300 + n, n, max(pages, 1), pad_every=pad)
    d = kstore_to_device(ks)
    pages = torch.zeros((ks.num_pages, fp4idx.FP8_PAGE_BYTES), dtype=torch.uint8, device="cuda")
    fp4idx.store_k_fp8(d["k"], d["positions"], d["slots"], d["norm_w"], ks.eps, cs_dev, pages)
    ref, st = oracle.store_k_fp8(ks, cs)
    assert st == 0
    torch.cuda.synchronize()
    got = pages.cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        raise AssertionError("fp8 mismatch at %d bytes, first %s" % (len(bad), bad[0]))


@pytest.mark.parametrize("T", [1, 64, 1536])
def test_quant_q_decode_shapes(fx, T):
    """Query rows of the tiny, batch-64 and draft-256x6 decode workloads."""
    fp4idx, cs, cs_dev = fx
    from tests.gpu_util import bf16, dev
    rng = np.random.default_rng(T)
    q = wl._normal_bf16(rng, (T, 64, 128), rng.choice(128, 4, replace=False))
    pos = rng.integers(0, cs.shape[0], T).astype(np.int32)
    pos[0] = 0
    pos[-1] = cs.shape[0] - 1
    qp, qs = fp4idx.alloc_query(T)
    fp4idx.quant_q(bf16(q), dev(pos), cs_dev, qp, qs)
    ref_p, ref_s, st = oracle.quant_q(q, pos, cs)
    assert st == 0
    _assert_cache_equal(qp.cpu().numpy(), qs.cpu().numpy(), ref_p, ref_s)


def test_quant_q_prefill_rows(fx):
    fp4idx, cs, cs_dev = fx
    from tests.gpu_util import bf16, dev
    rng = np.random.default_rng(1)
    T = 8192
    q = wl._normal_bf16(rng, (T, 64, 128))
    pos = (61440 + np.arange(T)).astype(np.int32)
    qp, qs = fp4idx.alloc_query(T)
    fp4idx.quant_q(bf16(q), dev(pos), cs_dev, qp, qs)
    sample = rng.choice(T, 256, replace=False)
    ref_p, ref_s, st = oracle.quant_q(q[sample], pos[sample], cs)
    assert st == 0
    _assert_cache_equal(qp.cpu().numpy()[sample], qs.cpu().numpy()[sample], ref_p, ref_s)


def test_api_rejects_bad_arguments(fx):
    fp4idx, cs, cs_dev = fx
    from tests.gpu_util import bf16, dev
    q = torch.zeros((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    qp, qs = fp4idx.alloc_query(2)
    with pytest.raises(fp4idx.Fp4IdxError) as e:
        fp4idx.quant_q(q, dev(np.zeros(2, np.int32)), cs_dev, qp, qs)
    assert e.value.code == 2
