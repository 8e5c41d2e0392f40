"""GPU top-k on given logits: the selection must be exactly the k largest values
(ties to the lower positions), in ascending position order, -1 padded.  Covers every
path of the kernel: spread values (bucket + rank), heavy tails, many duplicates and
all-equal rows (radix fallback), rows longer than the shared-memory cache."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def expected(lg, L, k):
    """The oracle's selection of the row's first L values (float32 values are exact in
    its float64, so equal values stay equal and go to the lower positions)."""
    return oracle.topk(np.asarray(lg[:L], np.float64), L, k)


def run(rows, lens, k, stride=None):
    from sparse_attention_fp4_gb300 import fp4idx
    T = len(rows)
    Lmax = max(1, max(lens))
    stride = stride or Lmax
    buf = np.full((T, stride), np.nan, np.float32)
    for t, r in enumerate(rows):
        buf[t, :lens[t]] = r[:lens[t]]
    lg = torch.from_numpy(buf).cuda()
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.empty((T, k), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(fp4idx.topk_workspace_bytes(T, Lmax), dtype=torch.uint8, device="cuda")
    fp4idx.topk(lg, cl, Lmax, k, ws, out, status=status)
    torch.cuda.synchronize()
    assert fp4idx.read_status(status) == 0
    return out.cpu().numpy()


def _dist(rng, kind, L):
    if kind == "normal":
        return rng.standard_normal(L).astype(np.float32)
    if kind == "cauchy":
        return rng.standard_cauchy(L).astype(np.float32)
    if kind == "outliers":
        x = rng.standard_normal(L).astype(np.float32)
        x[rng.choice(L, min(5, L), replace=False)] = np.float32(1e6)
        return x
    if kind == "dups":
        return np.round(rng.standard_normal(L) * 4).astype(np.float32) + np.float32(0.5)
    if kind == "equal":
        return np.full(L, 3.25, np.float32)
    if kind == "positive_narrow":
        return (100 + rng.random(L) * 1e-3).astype(np.float32)
    if kind == "signed_zeros":  # -0 and +0 are equal values: ties go to the lower positions
        x = np.where(rng.random(L) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        x[rng.random(L) < 0.01] = np.float32(1.0)
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "cauchy", "outliers", "dups", "equal", "positive_narrow", "signed_zeros"])
@pytest.mark.parametrize("stride_pad", [0, 3])
def test_topk_distributions(kind, stride_pad):
    rng = np.random.default_rng(hash(kind) % 1000)
    lens = [0, 1, 2047, 2048, 2049, 4096, 21000, 32768]
    rows = [_dist(rng, kind, max(L, 1)) for L in lens]
    k = 2048
    got = run(rows, lens, k, stride=max(lens) + stride_pad)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, k)), (kind, t, L)


def test_topk_long_rows_outside_the_cache():
    rng = np.random.default_rng(5)
    lens = [49152, 50000, 65536]
    rows = [_dist(rng, kd, L) for kd, L in zip(["normal", "dups", "cauchy"], lens)]
    got = run(rows, lens, 4096)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, 4096)), t


@pytest.mark.parametrize("k", [1, 7, 512, 4096])
def test_topk_small_and_max_k(k):
    rng = np.random.default_rng(k)
    lens = [1, 100, 5000, 17000]
    rows = [_dist(rng, "normal", L) for L in lens]
    got = run(rows, lens, k)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, k)), (k, t)


@pytest.mark.parametrize("kind", ["normal", "dups"])
def test_topk_chunk_boundaries(kind):
    rng = np.random.default_rng(11)
    lens = [2049, 4095, 4096, 4097, 8191, 8192, 8193, 12289, 65535]
    rows = [_dist(rng, kind, L) for L in lens]
    got = run(rows, lens, 2048, stride=65536 + 1)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, 2048)), (kind, t, L)


@pytest.mark.parametrize("longest", [8191, 8192, 8193])
def test_topk_pair_threshold(longest):
    """Few rows: one CTA per row while the longest row has at most 8,192 positions, a CTA
    pair per row past that; the rows around the switch select the same either way."""
    rng = np.random.default_rng(longest)
    lens = [longest, 2049, 4097, 8000, 3000]
    rows = [_dist(rng, kd, L) for kd, L in zip(["normal", "dups", "cauchy", "outliers", "normal"], lens)]
    got = run(rows, lens, 2048)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, 2048)), (longest, t, L)


@pytest.mark.parametrize("kind", ["normal", "dups", "signed_zeros"])
def test_topk_many_rows(kind):
    """More rows than SMs: one CTA of 512 threads per row, two of them an SM.  Lengths from
    empty to past the keys a CTA keeps in shared memory."""
    rng = np.random.default_rng(13 + len(kind))
    lens = [int(x) for x in rng.integers(0, 40000, size=194)] + [0, 1, 2047, 2048, 2049, 65535]
    rows = [_dist(rng, kind, max(L, 1)) for L in lens]
    got = run(rows, lens, 2048)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, 2048)), (kind, t, L)


def _sample_positions(L, n=1024):
    return (np.arange(n, dtype=np.int64) * L) // n


def test_topk_rows_that_mislead_the_sample():
    """Rows whose strided sample (every L/1024-th position) spreads far wider or far
    narrower than the rest of the row: a selection that estimated its threshold from such
    a sample would keep too few or too many candidates.  The exact radix selection has no
    sample; these rows stay as adversarial cases for any later change that adds one."""
    rng = np.random.default_rng(12)
    lens = [32768, 20000, 32768, 9000]
    rows = []
    for i, L in enumerate(lens):
        sp = _sample_positions(L)
        if i % 2 == 0:  # sample spread over [0, 100], every other logit in [0, 1)
            x = rng.random(L).astype(np.float32)
            x[sp] = np.linspace(0, 100, sp.size, dtype=np.float32)
        else:  # sample spread over [0, 1], every other logit just below its top
            x = (0.99 + 0.001 * rng.random(L)).astype(np.float32)
            x[sp] = np.linspace(0, 1, sp.size, dtype=np.float32)
        rows.append(x)
    got = run(rows, lens, 2048)
    for t, L in enumerate(lens):
        assert np.array_equal(got[t], expected(rows[t], L, 2048)), t


def _boundary_row(rng, L, k, n_band, band):
    """k - 2 keys at 10, n_band keys whose values share the top 22 key bits (the values in
    `band`), the rest at 1; shuffled.  With n_band == 2 the boundary sub-bin is taken whole;
    with n_band == 3 one of its keys must be left out (the higher position)."""
    x = np.full(L, 1.0, np.float32)
    pos = rng.permutation(L)
    x[pos[:k - 2]] = 10.0
    x[pos[k - 2:k - 2 + n_band]] = np.asarray(band[:n_band], np.float32)
    return x


# a CTA pair per row (few rows longer than 8,192); one CTA per row (few short rows, or
# more than half the SMs); more rows than SMs: one 512-thread CTA per row
@pytest.mark.parametrize("n_rows,L", [(8, 16384), (8, 4096), (100, 4096), (200, 4096)])
@pytest.mark.parametrize("n_band,band", [(2, [5.0, 5.0]), (2, [5.0, 5.0000005]), (3, [5.0, 5.0, 5.0]),
                                         (3, [5.0000005, 5.0, 5.0000005])])
def test_topk_boundary_sub_bin(n_rows, L, n_band, band):
    rng = np.random.default_rng(21 + n_band)
    k = 2048
    lens = [L] * n_rows
    rows = [_boundary_row(rng, L, k, n_band, band) for _ in range(n_rows)]
    got = run(rows, lens, k)
    for t in range(n_rows):
        assert np.array_equal(got[t], expected(rows[t], L, k)), (n_rows, n_band, t)
