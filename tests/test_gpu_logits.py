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


@pytest.mark.parametrize("seed,lens,rps,k,zeros", SMALL)
def test_small_batches_against_oracle(cs, seed, lens, rps, k, zeros):
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=k, zero_rows=zeros)
    got = run_gpu_indexer(b, cs)
    assert got["status"] == 0
    ref = oracle.run_indexer(b, cs)
    assert np.array_equal(got["payload"].cpu().numpy(), ref["payload"])
    assert np.array_equal(got["q_payload"].cpu().numpy(), ref["q_payload"])
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
