"""Failure detection of the logits kernels' bounded waits, with no GPU fault: the test
switch tells the producer warps to issue nothing, so the first wait of every other role
runs out after a short limit.  The launch must record FP4IDX_ERR_TIMEOUT in the status
word and return (the copies it issued landed, its tensor memory freed), and the context
must stay usable: with the switch off, the next calls are parity-green again."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import bf16, check_logits, check_topk, dev, run_gpu_indexer

pytestmark = pytest.mark.gpu

TIMEOUT = 6
LIMIT_NS = 5_000_000  # 5 ms a wait


@pytest.fixture
def waits_restored():
    from sparse_attention_fp4_gb300 import fp4idx
    yield fp4idx
    fp4idx.test_pipeline_waits(False, 0)


def _check_batch(b, cs, got):
    assert got["status"] == 0
    ref = oracle.run_indexer(b, cs)
    for t in range(b.n_rows):
        L = int(b.context_lens[t])
        check_logits(got["logits"][t], ref["logits"][t], ref["bound"][t], L, "row %d" % t)
        check_topk(got["topk"][t], ref["logits"][t], ref["bound"][t], L, b.topk, "row %d" % t)


@pytest.mark.parametrize("fused", [False, True], ids=["two_launches", "fused"])
def test_fp4_logits_wait_runs_out_then_recovers(cs, waits_restored, fused):
    fp4idx = waits_restored
    b = wl.small_batch(60, [3000, 700, 64], rows_per_seq=2, topk=128)
    fp4idx.test_pipeline_waits(True, LIMIT_NS)
    stalled = run_gpu_indexer(b, cs, fused=fused)
    assert stalled["status"] == TIMEOUT
    fp4idx.test_pipeline_waits(False, 0)
    # the same cache and a fresh schedule: the context is intact and the result exact
    _check_batch(b, cs, run_gpu_indexer(b, cs, payload=stalled["payload"], scale=stalled["scale"], fused=fused))


def test_fp8_logits_wait_runs_out_then_recovers(cs, waits_restored):
    fp4idx = waits_restored
    b = wl.small_batch(61, [2000, 130], rows_per_seq=1, topk=64)
    ks = b.kstore
    T = b.n_rows
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs_dev = bf16(cs)
    pages = torch.zeros((b.num_pages, fp4idx.FP8_PAGE_BYTES), dtype=torch.uint8, device="cuda")
    fp4idx.store_k_fp8(bf16(ks.k_rows), dev(ks.positions), dev(ks.slots), bf16(ks.norm_w), ks.eps, cs_dev, pages,
                       status=status)
    q8 = torch.empty((T, 8, 64, 16), dtype=torch.uint8, device="cuda")
    s8 = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    fp4idx.quant_q_fp8(bf16(b.q), dev(b.q_positions), cs_dev, q8, s8, status=status)
    cl, rs, pt = dev(b.context_lens), dev(b.row_seq), dev(b.page_table)
    Lmax = int(b.context_lens.max())
    sched = torch.empty(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    fp4idx.build_schedule(cl, rs, sched)
    assert fp4idx.read_status(status) == 0

    def run():
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lg = torch.full((T, Lmax), float("nan"), dtype=torch.float32, device="cuda")
        fp4idx.logits_fp8(q8, s8, dev(b.w), pages, pt, rs, cl, Lmax, sched, lg, status=st)
        return fp4idx.read_status(st), lg.cpu().numpy()

    fp4idx.test_pipeline_waits(True, LIMIT_NS)
    st, _ = run()
    assert st == TIMEOUT
    fp4idx.test_pipeline_waits(False, 0)
    st, lg = run()
    assert st == 0
    ref, bnd, rst = oracle.logits_fp8(q8.cpu().numpy(), s8.cpu().numpy(), b.w, pages.cpu().numpy(), b.page_table,
                                      b.row_seq, b.context_lens)
    assert rst == 0
    for t in range(T):
        L = int(b.context_lens[t])
        check_logits(lg[t], ref[t], bnd[t], L, "fp8 row %d" % t)


@pytest.fixture(scope="module")
def cs():
    return wl.rope_cos_sin_table()
