"""fp4idx_prepare_step: the schedule build, the K store and the Q quant in one launch must
give the bytes of the three separate calls (and, for the cache and the queries, of the
oracle), on ragged batches with padding slots, on more rows than one block scans at once,
and followed by the logits + top-k call."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import bf16, check_topk, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cs():
    return wl.rope_cos_sin_table()


def _both(b, cs, n_new_rows):
    """The step preparation of a batch two ways: fp4idx_prepare_step, and the three calls.
    The cache first holds every K row but the last n_new_rows, which the step stores."""
    from sparse_attention_fp4_gb300 import fp4idx
    ks = b.kstore
    n_old = ks.n_rows - n_new_rows
    cs_dev = bf16(cs)
    out = []
    for joint in (True, False):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        payload, scale = fp4idx.alloc_cache(b.num_pages)
        if n_old > 0:
            fp4idx.store_k(bf16(ks.k_rows[:n_old]), dev(ks.positions[:n_old]), dev(ks.slots[:n_old]), bf16(ks.norm_w),
                           ks.eps, cs_dev, payload, scale, status=status)
        new = dict(k=bf16(ks.k_rows[n_old:]), pos=dev(ks.positions[n_old:]), slots=dev(ks.slots[n_old:]))
        T = b.n_rows
        qp = torch.zeros((T, 4, 64, 16), dtype=torch.uint8, device="cuda")
        qs = torch.zeros((T, 4, 64), dtype=torch.uint8, device="cuda")
        cl, rs = dev(b.context_lens), dev(b.row_seq)
        sched = torch.zeros(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
        if joint:
            fp4idx.prepare_step(new["k"], new["pos"], new["slots"], bf16(ks.norm_w), ks.eps, bf16(b.q),
                                dev(b.q_positions), cs_dev, payload, scale, qp, qs, cl, rs, sched, status=status)
        else:
            fp4idx.build_schedule(cl, rs, sched)
            fp4idx.store_k(new["k"], new["pos"], new["slots"], bf16(ks.norm_w), ks.eps, cs_dev, payload, scale,
                           status=status)
            fp4idx.quant_q(bf16(b.q), dev(b.q_positions), cs_dev, qp, qs, status=status)
        torch.cuda.synchronize()
        out.append(dict(status=fp4idx.read_status(status), payload=payload, scale=scale, qp=qp, qs=qs, sched=sched,
                        cl=cl, rs=rs))
    return out


@pytest.mark.parametrize("seed,lens,rps,n_new", [
    (70, [300, 64, 1, 129], 1, 4),
    (71, [2000, 5, 700, 64, 1500], 3, 5),
    (72, [0, 100, 0, 40], 1, 2),
    (73, [4096] * 40, 1, 40),
])
def test_prepare_step_equals_the_three_calls(cs, seed, lens, rps, n_new):
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=64, zero_rows=(0,) if seed == 72 else ())
    j, s = _both(b, cs, min(n_new, b.kstore.n_rows))
    assert j["status"] == 0 and s["status"] == 0
    for key in ("payload", "scale", "qp", "qs", "sched"):
        assert torch.equal(j[key], s[key]), key
    # and the cache and the queries are the oracle's
    payload, scale, st = oracle.store_k(b.kstore, cs)
    assert st == 0
    assert np.array_equal(j["payload"].cpu().numpy(), payload) and np.array_equal(j["scale"].cpu().numpy(), scale)
    qp, qs, st = oracle.quant_q(b.q, b.q_positions, cs)
    assert np.array_equal(j["qp"].cpu().numpy(), qp) and np.array_equal(j["qs"].cpu().numpy(), qs)


def test_prepare_step_schedule_past_one_chunk(cs):
    """1,536 draft rows: the 256-thread build walks six chunks of rows."""
    b = wl.draft_batch256()
    from sparse_attention_fp4_gb300 import fp4idx
    T = b.n_rows
    cl, rs = dev(b.context_lens), dev(b.row_seq)
    a = torch.zeros(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    c = torch.zeros_like(a)
    fp4idx.build_schedule(cl, rs, a)
    z = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    zi = torch.zeros(0, dtype=torch.int32, device="cuda")
    payload, scale = fp4idx.alloc_cache(1)
    qp, qs = fp4idx.alloc_query(T)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.prepare_step(z, zi, zi, bf16(b.kstore.norm_w), b.kstore.eps, bf16(b.q), dev(b.q_positions), bf16(cs),
                        payload, scale, qp, qs, cl, rs, c, status=status)
    torch.cuda.synchronize()
    assert fp4idx.read_status(status) == 0
    assert torch.equal(a, c)


@pytest.mark.parametrize("fused", [False, True], ids=["two_launches", "fused"])
def test_prepare_step_then_selection(cs, fused):
    """The whole step as the bench runs it (preparation, then the read side right behind it
    on the stream), against the oracle."""
    from sparse_attention_fp4_gb300 import fp4idx
    b = wl.small_batch(74, [3000, 700, 64, 2500], rows_per_seq=2, topk=256)
    j, _ = _both(b, cs, 4)
    assert j["status"] == 0
    T = b.n_rows
    Lmax = int(b.context_lens.max())
    lg = torch.full((T, Lmax), float("nan"), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, b.topk), dtype=torch.int32, device="cuda")
    ws = torch.empty(fp4idx.logits_workspace_bytes(T, Lmax, b.topk), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.logits_topk(j["qp"], j["qs"], dev(b.w), j["payload"], j["scale"], dev(b.page_table), j["rs"], j["cl"], Lmax,
                       b.topk, j["sched"], ws, topk, logits_out=lg, status=status, fused=fused)
    torch.cuda.synchronize()
    assert fp4idx.read_status(status) == 0
    ref = oracle.run_indexer(b, cs)
    got = topk.cpu().numpy()
    for t in range(T):
        check_topk(got[t], ref["logits"][t], ref["bound"][t], int(b.context_lens[t]), b.topk, "row %d" % t)
