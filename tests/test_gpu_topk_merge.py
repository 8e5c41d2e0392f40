"""Context-parallel top-k on the GPU, emulated with N logical shards of each row: every
shard selects from its own token range (fp4idx_topk on its own buffer, as one GPU of a
sharded run would), its values are gathered (fp4idx_topk_values), and fp4idx_topk_merge
combines the candidates.  The result must be exactly the selection of fp4idx_topk on the
whole row, ties included."""
import numpy as np
import pytest
import torch

from tests.gpu_util import dev, host
from tests.test_gpu_topk import _dist, expected

pytestmark = pytest.mark.gpu


def sharded_topk(rows, lens, k, bounds):
    """Per shard [lo, hi): its logits in a buffer of its own, its top-k, the values, and
    the global positions; then the merge."""
    from sparse_attention_fp4_gb300 import fp4idx
    T = len(rows)
    S = len(bounds) - 1
    cand_v = np.zeros((T, S, k), np.float32)
    cand_i = np.full((T, S, k), -1, np.int32)
    for s in range(S):
        lo, hi = bounds[s], bounds[s + 1]
        width = max(1, hi - lo)
        buf = np.full((T, width), np.nan, np.float32)
        slen = np.zeros(T, np.int32)
        for t in range(T):
            n = int(np.clip(lens[t] - lo, 0, hi - lo))
            slen[t] = n
            buf[t, :n] = rows[t][lo:lo + n]
        lg = dev(buf)
        cl = dev(slen)
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        ws = torch.empty(fp4idx.topk_workspace_bytes(T, width), dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4idx.topk(lg, cl, width, k, ws, idx, status=status)
        vals = torch.empty((T, k), dtype=torch.float32, device="cuda")
        fp4idx.topk_values(lg, idx, vals)
        assert fp4idx.read_status(status) == 0
        i_h = host(idx)
        cand_v[:, s] = host(vals)
        cand_i[:, s] = np.where(i_h >= 0, i_h + lo, -1)
    out = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(fp4idx.topk_merge_workspace_bytes(T, S, k), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.topk_merge(dev(cand_v), dev(cand_i), ws, out, status=status)
    assert fp4idx.read_status(status) == 0
    return host(out), cand_v, cand_i


@pytest.mark.parametrize("kind", ["normal", "dups", "equal", "cauchy", "signed_zeros"])
@pytest.mark.parametrize("bounds", [[0, 9000, 20000, 32768], [0, 1, 2048, 2049, 32768], [0, 16384, 32768]])
def test_sharded_selection_equals_whole_row(kind, bounds):
    rng = np.random.default_rng(hash((kind, len(bounds))) % 1000)
    lens = [0, 100, 2048, 2049, 5000, 20000, 32768]
    rows = [_dist(rng, kind, max(L, 1)) for L in lens]
    k = 2048
    got, cand_v, cand_i = sharded_topk(rows, lens, k, bounds)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, k)), (kind, bounds, t, L)
    # the gathered values are the rows' own values at the shards' selections
    for t in range(len(lens)):
        sel = cand_i[t] >= 0
        assert np.array_equal(cand_v[t][sel], rows[t][cand_i[t][sel]])


@pytest.mark.parametrize("k", [1, 7, 4096])
def test_sharded_selection_small_and_large_k(k):
    rng = np.random.default_rng(k)
    lens = [1, 300, 9000, 16000]
    rows = [_dist(rng, "dups", L) for L in lens]
    got, _, _ = sharded_topk(rows, lens, k, [0, 4000, 8000, 12000, 16000])
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, k)), (k, t)
