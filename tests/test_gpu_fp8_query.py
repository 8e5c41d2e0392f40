"""GPU FP8 query pack (the query side of the 132 B/token comparison path): the e4m3 bytes
and the fp32 scales equal the oracle's bit for bit; zero rows get scale 1 and +-0 codes; a
position outside the RoPE table is reported and its row left unwritten."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_fp4_gb300 import workloads as wl
from tests.gpu_util import bf16, dev, host

pytestmark = pytest.mark.gpu


def run(q, qpos, cs_np, fill=0xEE):
    from sparse_attention_fp4_gb300 import fp4idx
    T = q.shape[0]
    q8 = torch.full((T, 8, 64, 16), fill, dtype=torch.uint8, device="cuda")
    s8 = torch.full((T, 64), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4idx.quant_q_fp8(bf16(q), dev(qpos), bf16(cs_np), q8, s8, status=status)
    return host(q8), host(s8), fp4idx.read_status(status)


@pytest.mark.parametrize("seed,T", [(1, 1), (2, 7), (3, 64)])
def test_fp8_query_pack_matches_oracle(seed, T):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, 64, 128)).astype(np.float32)
    x[:, :, rng.choice(128, 4, replace=False)] *= 8.0  # outlier channels
    q = wl.f32_to_bf16_bits(x)
    if T > 1:
        q[1] = 0  # a zero row: scale 1, zero codes
    qpos = rng.integers(0, 131072, size=T).astype(np.int32)
    cs = wl.rope_cos_sin_table()
    q8, s8, st = run(q, qpos, cs)
    r8, rs8, rst = oracle.quant_q_fp8(q, qpos, cs)
    assert st == 0 and rst == 0
    assert np.array_equal(q8, r8)
    assert np.array_equal(s8.view(np.uint32), rs8.view(np.uint32))
    if T > 1:
        assert np.all(q8[1] & 0x7F == 0) and np.all(s8[1] == 1.0)  # +-0 (RoPE leaves some -0)


def test_bad_position_is_reported():
    rng = np.random.default_rng(9)
    q = wl.f32_to_bf16_bits(rng.standard_normal((2, 64, 128)).astype(np.float32))
    cs = wl.rope_cos_sin_table()
    qpos = np.array([5, cs.shape[0] + 3], np.int32)
    q8, s8, st = run(q, qpos, cs)
    assert st == 7  # FP4IDX_ERR_BAD_POSITION
    r8, rs8, _ = oracle.quant_q_fp8(q[:1], qpos[:1], cs)
    assert np.array_equal(q8[0], r8[0]) and np.all(q8[1] == 0xEE) and np.all(s8[1] == -1.0)
