"""GPU one-launch Q pack + head weights (fp4idx_quant_q_w): the packed queries are
byte-identical to fp4idx_quant_q's; the head weights are within the bound their fixed
summation order gives of the oracle's exact values, (hidden_dim/256 + 20) * 2^-24 *
|w_scale| * sum_d |hidden*w_proj| (a product meets at most 8*ceil(M/8) + 12 <=
hidden_dim/256 + 19 roundings, M = hidden_dim/256; bf16 products are exact in fp32); one-hot
rows come out exact; and a row's weights do not depend on the rows computed with it."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import bf16, dev, host

pytestmark = pytest.mark.gpu


def run(q, qpos, cs, hidden, w_proj, w_scale):
    from sparse_attention_fp4_gb300 import fp4idx
    T = q.shape[0]
    qp, qs = fp4idx.alloc_query(T)
    w_out = torch.full((T, 64), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.quant_q_w(bf16(q), dev(qpos), cs, bf16(hidden), bf16(w_proj), w_scale, qp, qs, w_out, status=status)
    assert fp4idx.read_status(status) == 0
    return host(qp), host(qs), host(w_out)


def inputs(seed, T, D):
    rng = np.random.default_rng(seed)
    q = wl.f32_to_bf16_bits(rng.standard_normal((T, 64, 128)).astype(np.float32))
    qpos = rng.integers(0, 4096, size=T).astype(np.int32)
    hidden = wl.f32_to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    w_proj = wl.f32_to_bf16_bits((rng.standard_normal((64, D)) / np.sqrt(D)).astype(np.float32))
    return q, qpos, hidden, w_proj


@pytest.mark.parametrize("T,D", [(1, 256), (5, 2048), (64, 7168), (3, 16384)])
def test_queries_and_head_weights(T, D):
    from sparse_attention_fp4_gb300 import fp4idx
    cs = bf16(wl.rope_cos_sin_table())
    q, qpos, hidden, w_proj = inputs(T * 7 + D, T, D)
    scale = 0.125
    qp, qs, w = run(q, qpos, cs, hidden, w_proj, scale)
    # the packed queries: byte-identical to the plain Q quant
    qp2, qs2 = fp4idx.alloc_query(T)
    fp4idx.quant_q(bf16(q), dev(qpos), cs, qp2, qs2)
    assert np.array_equal(qp, host(qp2)) and np.array_equal(qs, host(qs2))
    ref, bound = oracle.head_weights(hidden, w_proj, scale)
    tol = (D / 256 + 20) * 2.0 ** -24 * bound + 1e-30
    err = np.abs(w.astype(np.float64) - ref)
    assert np.all(err <= tol), (T, D, float((err / np.maximum(bound, 1e-30)).max()))


def test_one_hot_rows_are_exact():
    cs = bf16(wl.rope_cos_sin_table())
    T, D = 4, 1024
    q, qpos, _, w_proj = inputs(11, T, D)
    hidden = np.zeros((T, D), np.uint16)
    cols = [0, 31, 512, 1023]
    for t, d in enumerate(cols):
        hidden[t, d] = 0x3F80  # 1.0
    _, _, w = run(q, qpos, cs, hidden, w_proj, 0.5)
    ref, _ = oracle.head_weights(hidden, w_proj, 0.5)
    assert np.array_equal(w.astype(np.float64), ref)


def test_a_rows_weights_do_not_depend_on_the_batch():
    cs = bf16(wl.rope_cos_sin_table())
    T, D = 64, 7168
    q, qpos, hidden, w_proj = inputs(12, T, D)
    _, _, w_all = run(q, qpos, cs, hidden, w_proj, 1.0)
    for t in (0, 17, 63):
        _, _, w_one = run(q[t:t + 1], qpos[t:t + 1], cs, hidden[t:t + 1], w_proj, 1.0)
        assert np.array_equal(w_one[0], w_all[t]), t
