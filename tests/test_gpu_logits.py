"""GPU parity of the read side: schedule + paged-MQA logits (tcgen05 block-scaled FP4)
+ top-k against the CPU oracle, on small ragged cases and on the workload shapes."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import check_logits, check_topk, check_topk_self, run_gpu_indexer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cs():
    return wl.rope_cos_sin_table()


SMALL = [
    (1, [1], 1, 8, ()),
    (2, [63, 64, 65], 1, 16, ()),
    (3, [127, 128, 129, 130], 1, 32, ()),
    (4, [300, 1000, 5], 2, 64, ()),
    (5, [200, 61 + 64 * 3, 700], 6, 16, (3,)),
    (6, [0, 50, 0, 129], 1, 8, (0, 2)),
    (7, [2000, 2500, 1500, 2049], 3, 512, ()),
    (8, [4096] * 9, 1, 2048, ()),
    (9, [900], 8, 100, ()),
    (10, [700, 800], 9, 100, ()),          # 9 rows per sequence: a group boundary inside a run
    (11, [5000, 33, 7000, 1, 64], 1, 4096, (1,)),
]


@pytest.mark.parametrize("fused", [False, True], ids=["two_launches", "fused"])
@pytest.mark.parametrize("seed,lens,rps,k,zeros", SMALL)
def test_small_batches_against_oracle(cs, seed, lens, rps, k, zeros, fused):
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=k, zero_rows=zeros)
    got = run_gpu_indexer(b, cs, fused=fused)
    assert got["status"] == 0
    ref = oracle.run_indexer(b, cs)
    assert np.array_equal(got["payload"].cpu().numpy(), ref["payload"])
    assert np.array_equal(got["scale"].cpu().numpy(), ref["scale"])
    assert np.array_equal(got["q_payload"].cpu().numpy(), ref["q_payload"])
    assert np.array_equal(got["q_scale"].cpu().numpy(), ref["q_scale"])
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], ref["logits"][t], ref["bound"][t], L, "row %d" % t)
        check_topk(got["topk"][t], ref["logits"][t], ref["bound"][t], L, k, "row %d" % t)
        check_topk_self(got["topk"][t], got["logits"][t], L, k, "row %d" % t)


def test_workspace_path_matches_logits_out_path(cs):
    b = wl.small_batch(40, [3000, 700, 1, 2500], rows_per_seq=2, topk=256)
    a = run_gpu_indexer(b, cs, with_logits=True)
    w = run_gpu_indexer(b, cs, with_logits=False)
    assert a["status"] == 0 and w["status"] == 0
    assert np.array_equal(a["topk"], w["topk"])


def test_page_layout_and_batch_invariance(cs):
    """Identical logits (bit for bit) when the pages move and when a row runs alone."""
    b = wl.small_batch(41, [1500, 640, 2300], rows_per_seq=2, topk=128)
    base = run_gpu_indexer(b, cs)
    rng = np.random.default_rng(1)
    perm = rng.permutation(b.num_pages).astype(np.int32)
    P = base["payload"]
    S = base["scale"]
    P2 = torch.empty_like(P)
    S2 = torch.empty_like(S)
    inv = torch.from_numpy(perm).long().cuda()
    P2[inv] = P
    S2[inv] = S
    pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    moved = run_gpu_indexer(b, cs, page_table=pt2, payload=P2, scale=S2)
    assert moved["status"] == 0
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        assert np.array_equal(moved["logits"][t, :L], base["logits"][t, :L])
    assert np.array_equal(moved["topk"], base["topk"])
    # row 3 alone (its sequence keeps the same page-table row)
    import copy
    one = copy.copy(b)
    one.q = b.q[3:4]
    one.q_positions = b.q_positions[3:4]
    one.w = b.w[3:4]
    one.row_seq = b.row_seq[3:4]
    one.context_lens = b.context_lens[3:4]
    alone = run_gpu_indexer(one, cs, payload=P, scale=S)
    L = int(b.context_lens[3])
    assert np.array_equal(alone["logits"][0, :L], base["logits"][3, :L])
    assert np.array_equal(alone["topk"][0], base["topk"][3])


def test_repeat_runs_are_bitwise_identical(cs):
    b = wl.small_batch(42, [4000, 3000, 100, 2000], rows_per_seq=3, topk=300)
    r1 = run_gpu_indexer(b, cs)
    r2 = run_gpu_indexer(b, cs, payload=r1["payload"], scale=r1["scale"])
    assert np.array_equal(r1["logits"], r2["logits"], equal_nan=True)
    assert np.array_equal(r1["topk"], r2["topk"])


def test_bad_page_is_reported_not_faulted(cs):
    b = wl.small_batch(43, [500, 300], rows_per_seq=1, topk=32)
    pt = b.page_table.copy()
    pt[1, 2] = b.num_pages + 1000
    got = run_gpu_indexer(b, cs, page_table=pt)
    assert got["status"] == 5
    ref = oracle.run_indexer(b, cs)
    L = int(b.context_lens[0])
    check_logits(got["logits"][0], ref["logits"][0], ref["bound"][0], L, "intact row")


def _sampled_rows(b, n, rng, must=()):
    cand = np.arange(b.n_rows)
    pick = set(rng.choice(cand, min(n, cand.size), replace=False).tolist())
    pick.update(must)
    return np.array(sorted(pick))


@pytest.mark.parametrize("maker,nsample", [(wl.tiny_decode, 1), (wl.decode_batch64, 6), (wl.draft_batch256, 16),
                                           (wl.prefill_chunk, 10)])
def test_workloads_against_oracle(cs, maker, nsample):
    b = maker()
    got = run_gpu_indexer(b, cs)
    assert got["status"] == 0
    payload, scale, st = oracle.store_k(b.kstore, cs)
    assert st == 0
    assert np.array_equal(got["payload"].cpu().numpy(), payload) and np.array_equal(got["scale"].cpu().numpy(), scale)
    rng = np.random.default_rng(7)
    must = [0, b.n_rows - 1]
    if b.n_rows > 48:
        must += [b.n_rows - 48, 8 * 6]  # a padded row and a page-crossing draft row (draft workload)
    rows = _sampled_rows(b, nsample, rng, must)
    qp, qs, st = oracle.quant_q(b.q[rows], b.q_positions[rows], cs)
    assert np.array_equal(got["q_payload"].cpu().numpy()[rows], qp)
    lg, bnd, st = oracle.logits(qp, qs, b.w[rows], payload, scale, b.page_table, b.row_seq[rows],
                                b.context_lens[rows])
    assert st == 0
    for i, t in enumerate(rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], lg[i], bnd[i], L, "%s row %d" % (b.name, t))
        check_topk(got["topk"][t], lg[i], bnd[i], L, b.topk, "%s row %d" % (b.name, t))
    self_rows = np.arange(b.n_rows) if b.n_rows <= 2048 else _sampled_rows(b, 512, rng, must)
    for t in self_rows:
        check_topk_self(got["topk"][t], got["logits"][t], int(b.context_lens[t]), b.topk, "%s row %d" % (b.name, t))


def _read_side(b, cs, payload, scale, sched=None, separate=False, k=None):
    """The read side alone on a stored cache: Q quant, schedule (unless given), then either
    the fused call (fp4idx_logits_topk_fused) or the two separate calls (fp4idx_logits,
    then fp4idx_topk).  Returns (status, logits, topk)."""
    from sparse_attention_fp4_gb300 import fp4idx
    from tests.gpu_util import bf16, dev
    k = b.topk if k is None else k
    T = b.n_rows
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qp, qs = fp4idx.alloc_query(T)
    fp4idx.quant_q(bf16(b.q), dev(b.q_positions), bf16(cs), qp, qs, status=status)
    cl, rs, pt = dev(b.context_lens), dev(b.row_seq), dev(b.page_table)
    Lmax = int(max(1, b.context_lens.max()))
    if sched is None:
        sched = torch.empty(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
        fp4idx.build_schedule(cl, rs, sched)
    lg = torch.full((T, Lmax), float("nan"), dtype=torch.float32, device="cuda")
    topk = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    if separate:
        fp4idx.logits(qp, qs, dev(b.w), payload, scale, pt, rs, cl, Lmax, sched, lg, status=status)
        ws = torch.empty(fp4idx.topk_workspace_bytes(T, Lmax), dtype=torch.uint8, device="cuda")
        fp4idx.topk(lg, cl, Lmax, k, ws, topk, status=status)
    else:
        ws = torch.empty(fp4idx.logits_workspace_bytes(T, Lmax, k), dtype=torch.uint8, device="cuda")
        fp4idx.logits_topk(qp, qs, dev(b.w), payload, scale, pt, rs, cl, Lmax, k, sched, ws, topk, logits_out=lg,
                           status=status, fused=True)
    torch.cuda.synchronize()
    return fp4idx.read_status(status), lg.cpu().numpy(), topk.cpu().numpy()


def _stored(b, cs):
    from sparse_attention_fp4_gb300 import fp4idx
    from tests.gpu_util import bf16, dev
    ks = b.kstore
    payload, scale = fp4idx.alloc_cache(b.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.store_k(bf16(ks.k_rows), dev(ks.positions), dev(ks.slots), bf16(ks.norm_w), ks.eps, bf16(cs), payload,
                   scale, status=status)
    assert fp4idx.read_status(status) == 0
    return payload, scale


@pytest.mark.parametrize("seed,lens,rps,k,zeros", [SMALL[3], SMALL[4], SMALL[5], SMALL[9], SMALL[10]])
def test_fused_selection_equals_separate_launches(cs, seed, lens, rps, k, zeros):
    """The logits launch's own selection (few rows) and the separate top-k launch select
    from bit-identical logits with the same rule, so they agree exactly."""
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=k, zero_rows=zeros)
    payload, scale = _stored(b, cs)
    st1, lg1, tk1 = _read_side(b, cs, payload, scale)
    st2, lg2, tk2 = _read_side(b, cs, payload, scale, separate=True)
    assert st1 == 0 and st2 == 0
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        assert np.array_equal(lg1[t, :L], lg2[t, :L]), t
    assert np.array_equal(tk1, tk2)


def test_schedule_reused_across_calls(cs):
    """A schedule built once serves several fused calls in a row (as every layer of a
    forward would use it): each call counts its groups complete and leaves the counters at
    zero for the next."""
    from sparse_attention_fp4_gb300 import fp4idx
    from tests.gpu_util import dev
    b = wl.small_batch(44, [3000, 129, 5000, 64, 2100], rows_per_seq=3, topk=256, zero_rows=(4,))
    payload, scale = _stored(b, cs)
    sched = torch.empty(fp4idx.schedule_workspace_bytes(b.n_rows), dtype=torch.uint8, device="cuda")
    fp4idx.build_schedule(dev(b.context_lens), dev(b.row_seq), sched)
    runs = [_read_side(b, cs, payload, scale, sched=sched) for _ in range(3)]
    ref = oracle.run_indexer(b, cs)
    for st, lg, tk in runs:
        assert st == 0
        assert np.array_equal(tk, runs[0][2])
        for t in range(b.n_rows):
            L = int(b.context_lens[t])
            check_topk(tk[t], ref["logits"][t], ref["bound"][t], L, b.topk, "row %d" % t)


def test_fused_selection_of_rows_past_shared_memory(cs):
    """Rows longer than the 32,768 sort keys a CTA keeps in shared memory spill the rest
    to the workspace; the fused selection still equals the oracle's."""
    b = wl.small_batch(45, [40000, 33000, 65536, 32769], rows_per_seq=1, topk=2048)
    # the decode query position 4L - 1 would pass the RoPE table for these lengths
    b.q_positions = np.minimum(b.q_positions, wl.ROPE_MAX_POS - 1).astype(np.int32)
    got = run_gpu_indexer(b, cs, fused=True)
    assert got["status"] == 0
    ref = oracle.run_indexer(b, cs)
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], ref["logits"][t], ref["bound"][t], L, "row %d" % t)
        check_topk(got["topk"][t], ref["logits"][t], ref["bound"][t], L, b.topk, "row %d" % t)
        check_topk_self(got["topk"][t], got["logits"][t], L, b.topk, "row %d" % t)


@pytest.mark.parametrize("rows", ["half", "half+1", "sms", "sms+1"])
def test_row_count_at_the_fused_limits(cs, rows):
    """The fused call at its limits: a CTA pair per row up to half as many rows as SMs, one
    CTA per row up to as many rows as SMs, the two launches beyond."""
    from sparse_attention_fp4_gb300 import fp4idx
    sms = fp4idx.num_sms()
    n = {"half": sms // 2, "half+1": sms // 2 + 1, "sms": sms, "sms+1": sms + 1}[rows]
    extra = n % 2
    rng = np.random.default_rng(46 + extra)
    lens = [int(x) for x in rng.integers(0, 3000, size=n)]
    b = wl.small_batch(46 + extra, lens, rows_per_seq=1, topk=300)
    got = run_gpu_indexer(b, cs, fused=True)
    assert got["status"] == 0
    ref = oracle.run_indexer(b, cs)
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_topk(got["topk"][t], ref["logits"][t], ref["bound"][t], L, b.topk, "row %d" % t)
        check_topk_self(got["topk"][t], got["logits"][t], L, b.topk, "row %d" % t)
