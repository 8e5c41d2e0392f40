"""GPU parity of the FP8 comparison path's logits (tensor-core e4m3 contraction over the
132 B/token fused pages): the cache and query bytes equal the oracle's, and the logits
agree with the oracle's binary64 FP8 logits within 1e-5 * sum_h |w q k| + 1e-6 on ragged
batches spanning several tiles, shared-sequence groups, zero-length rows, a bad page and
sampled rows of the decode batch."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import bf16, check_logits, check_topk, check_topk_self, dev, host

pytestmark = pytest.mark.gpu

UNWRITTEN = np.float32(np.inf)


@pytest.fixture(scope="module")
def cs():
    return wl.rope_cos_sin_table()


def run_fp8(b, cs_np, page_table=None, k=None):
    """FP8 K store, FP8 query pack, schedule and FP8 logits, all on the GPU; with k, the
    fused logits + top-k call instead (once with logits_out, once through the workspace)."""
    from sparse_attention_fp4_gb300 import fp4idx
    cs = bf16(cs_np)
    ks = b.kstore
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pages = torch.zeros((b.num_pages, fp4idx.FP8_PAGE_BYTES), dtype=torch.uint8, device="cuda")
    fp4idx.store_k_fp8(bf16(ks.k_rows), dev(ks.positions), dev(ks.slots), bf16(ks.norm_w), ks.eps, cs, pages,
                       status=status)
    T = b.n_rows
    q8 = torch.empty((T, 8, 64, 16), dtype=torch.uint8, device="cuda")
    s8 = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    fp4idx.quant_q_fp8(bf16(b.q), dev(b.q_positions), cs, q8, s8, status=status)
    cl, rs = dev(b.context_lens), dev(b.row_seq)
    Lmax = int(max(1, b.context_lens.max()))
    sched = torch.empty(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    fp4idx.build_schedule(cl, rs, sched)
    lg = torch.full((T, Lmax), float(UNWRITTEN), dtype=torch.float32, device="cuda")
    pt = dev(b.page_table if page_table is None else page_table)
    sel = sel_ws = None
    if k is None:
        fp4idx.logits_fp8(q8, s8, dev(b.w), pages, pt, rs, cl, Lmax, sched, lg, status=status)
    else:
        ws = torch.empty(fp4idx.logits_workspace_bytes(T, Lmax, k), dtype=torch.uint8, device="cuda")
        sel = torch.empty((T, k), dtype=torch.int32, device="cuda")
        sel_ws = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = dev(b.w)
        fp4idx.logits_topk_fp8(q8, s8, w, pages, pt, rs, cl, Lmax, k, sched, ws, sel, logits_out=lg, status=status)
        fp4idx.logits_topk_fp8(q8, s8, w, pages, pt, rs, cl, Lmax, k, sched, ws, sel_ws, status=status)
    torch.cuda.synchronize()
    return dict(status=fp4idx.read_status(status), pages=host(pages), q8=host(q8), s8=host(s8), logits=host(lg),
                topk=None if sel is None else host(sel), topk_ws=None if sel_ws is None else host(sel_ws))


def oracle_operands(b, cs_np):
    pages, st = oracle.store_k_fp8(b.kstore, cs_np)
    assert st == 0
    q8, s8, st = oracle.quant_q_fp8(b.q, b.q_positions, cs_np)
    assert st == 0
    return pages, q8, s8


def assert_same_operands(got, pages, q8, s8):
    assert np.array_equal(got["pages"], pages)
    assert np.array_equal(got["q8"], q8)
    assert np.array_equal(got["s8"].view(np.uint32), s8.view(np.uint32))


CASES = [
    (1, [1], 1, ()),
    (2, [63, 64, 65], 1, ()),
    (3, [127, 128, 129, 130], 1, ()),
    (4, [300, 1000, 5], 2, ()),
    (5, [200, 61 + 64 * 3, 700], 6, (3,)),
    (6, [0, 50, 0, 129], 1, (0, 2)),
    (7, [2000, 2500, 1500, 2049], 3, ()),
    (10, [700, 800], 9, ()),  # 9 rows per sequence: a group boundary inside a run
    (11, [5000, 33, 7000, 1, 64], 1, (1,)),
]


@pytest.mark.parametrize("seed,lens,rps,zeros", CASES)
def test_fp8_logits_against_oracle(cs, seed, lens, rps, zeros):
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=8, zero_rows=zeros)
    got = run_fp8(b, cs)
    assert got["status"] == 0
    pages, q8, s8 = oracle_operands(b, cs)
    assert_same_operands(got, pages, q8, s8)
    lg, bnd, st = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens)
    assert st == 0
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], lg[t], bnd[t], L, "fp8 row %d" % t)
        assert np.all(got["logits"][t, L:] == UNWRITTEN), "fp8 row %d: written past its context" % t


def test_fp8_bad_page_is_reported_and_marked(cs):
    b = wl.small_batch(43, [500, 300], rows_per_seq=1, topk=8)
    pt = b.page_table.copy()
    pt[1, 2] = b.num_pages + 1000  # row 1's tokens 128..191
    got = run_fp8(b, cs, page_table=pt)
    assert got["status"] == 5  # FP4IDX_ERR_BAD_PAGE
    pages, q8, s8 = oracle_operands(b, cs)
    lg, bnd, st = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens)
    assert st == 0
    check_logits(got["logits"][0], lg[0], bnd[0], int(b.context_lens[0]), "intact row")
    row = got["logits"][1]
    assert np.all(np.isnan(row[128:192]))
    keep = np.r_[0:128, 192:int(b.context_lens[1])]
    err = np.abs(row[keep].astype(np.float64) - lg[1][keep])
    assert np.all(err <= 1e-5 * bnd[1][keep] + 1e-6)


def test_fp8_decode_batch_sampled_rows(cs):
    b = wl.decode_batch64()
    got = run_fp8(b, cs)
    assert got["status"] == 0
    pages, q8, s8 = oracle_operands(b, cs)
    assert_same_operands(got, pages, q8, s8)
    rows = np.array([0, 17, b.n_rows - 1])
    lg, bnd, st = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens, rows=rows)
    assert st == 0
    for i, t in enumerate(rows):
        check_logits(got["logits"][t], lg[i], bnd[i], int(b.context_lens[t]), "decode fp8 row %d" % t)


@pytest.mark.parametrize("seed,lens,rps,k", [(21, [3000, 700, 1, 2500], 2, 256), (22, [5000, 33, 0, 64], 1, 2048),
                                             (23, [128, 129, 4100], 3, 100)])
def test_fp8_logits_topk_against_oracle(cs, seed, lens, rps, k):
    """The fused FP8 call: the k highest oracle logits (up to swaps within tolerance of the
    k-th), ascending, -1 padding; the same selection with and without logits_out."""
    b = wl.small_batch(seed, lens, rows_per_seq=rps, topk=k)
    got = run_fp8(b, cs, k=k)
    assert got["status"] == 0
    assert np.array_equal(got["topk"], got["topk_ws"])
    pages, q8, s8 = oracle_operands(b, cs)
    assert_same_operands(got, pages, q8, s8)
    lg, bnd, st = oracle.logits_fp8(q8, s8, b.w, pages, b.page_table, b.row_seq, b.context_lens)
    assert st == 0
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], lg[t], bnd[t], L, "fp8 row %d" % t)
        check_topk(got["topk"][t], lg[t], bnd[t], L, k, "fp8 row %d" % t)
        check_topk_self(got["topk"][t], got["logits"][t], L, k, "fp8 row %d" % t)
