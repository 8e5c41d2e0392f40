"""fp4idx_topk_noalloc, the top-k entry point whose scratch is the library's fixed
per-device array: the same selection as fp4idx_topk (which takes a workspace) on two
different calls in a row, at the limit and across it, where the call is refused before
anything is enqueued.  Collected last on purpose; it must also pass alone in a fresh
process, where its first call is the one that sets the array up."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _rows(rng, lens):
    rows = []
    for i, L in enumerate(lens):
        kind = i % 3
        if kind == 0:
            x = rng.standard_normal(max(L, 1))
        elif kind == 1:
            x = np.round(rng.standard_normal(max(L, 1)) * 4) + 0.5  # many ties
        else:
            x = rng.standard_cauchy(max(L, 1))
        rows.append(x.astype(np.float32))
    return rows


def _inputs(rows, lens, stride):
    buf = np.full((len(rows), stride), np.nan, np.float32)
    for t, r in enumerate(rows):
        buf[t, :lens[t]] = r[:lens[t]]
    lg = torch.from_numpy(buf).cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return lg, cl


def _expected(row, L, k):
    import oracle
    return oracle.topk(np.asarray(row[:L], np.float64), L, k)


def _with_workspace(lg, cl, Lmax, k):
    from sparse_attention_fp4_gb300 import fp4idx
    T = cl.numel()
    out = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(fp4idx.topk_workspace_bytes(T, Lmax), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.topk(lg, cl, Lmax, k, ws, out, status=status)
    assert fp4idx.read_status(status) == 0
    return out.cpu().numpy()


def _noalloc(lg, cl, Lmax, k):
    from sparse_attention_fp4_gb300 import fp4idx
    T = cl.numel()
    out = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.topk_noalloc(lg, cl, Lmax, k, out, status=status)
    assert fp4idx.read_status(status) == 0
    return out.cpu().numpy()


def test_noalloc_matches_workspace_topk_on_two_calls_in_a_row():
    rng = np.random.default_rng(77)
    k1, lens1 = 2048, [0, 1, 2047, 2049, 9000, 32768, 20000, 4096]
    k2, lens2 = 512, [600, 513, 100, 65536, 12345, 511]
    rows1, rows2 = _rows(rng, lens1), _rows(rng, lens2)
    lg1, cl1 = _inputs(rows1, lens1, max(lens1) + 3)
    lg2, cl2 = _inputs(rows2, lens2, max(lens2))
    got1 = _noalloc(lg1, cl1, max(lens1), k1)
    got2 = _noalloc(lg2, cl2, max(lens2), k2)  # second call in a row, another shape
    np.testing.assert_array_equal(got1, _with_workspace(lg1, cl1, max(lens1), k1))
    np.testing.assert_array_equal(got2, _with_workspace(lg2, cl2, max(lens2), k2))
    for t, L in enumerate(lens1):
        np.testing.assert_array_equal(got1[t], _expected(rows1[t], L, k1))
    for t, L in enumerate(lens2):
        np.testing.assert_array_equal(got2[t], _expected(rows2[t], L, k2))


def test_noalloc_limit():
    from sparse_attention_fp4_gb300 import fp4idx
    Lmax, k = 65536, 2048
    fits = 1
    while fp4idx.topk_workspace_bytes(fits + 1, Lmax) <= fp4idx.TOPK_NOALLOC_MAX_BYTES:
        fits += 1
    too_many = fits + 1
    assert fits >= 16
    rng = np.random.default_rng(78)
    lens = [int(v) for v in rng.integers(Lmax // 2, Lmax + 1, size=too_many)]
    lens[0] = Lmax
    rows = _rows(rng, lens)
    lg, cl = _inputs(rows, lens, Lmax)
    # the largest row count that fits runs and agrees with the workspace entry point
    got = _noalloc(lg[:fits], cl[:fits], Lmax, k)
    np.testing.assert_array_equal(got, _with_workspace(lg[:fits], cl[:fits], Lmax, k))
    # one more row is refused on the host, with nothing enqueued
    out = torch.full((too_many, k), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(fp4idx.Fp4IdxError) as err:
        fp4idx.topk_noalloc(lg, cl, Lmax, k, out)
    assert err.value.code == 10
    torch.cuda.synchronize()
    assert bool((out == -7).all())
