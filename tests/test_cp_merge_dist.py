"""The context-parallel exchange on CPU: two gloo ranks each own half of every row's
compressed tokens, select their shard's top-k with the oracle, all-gather the (value,
global position) candidates, and merge them.  Both ranks must end with exactly the
oracle's selection on the whole row."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(seed):
    rng = np.random.default_rng(seed)
    lens = [0, 50, 1000, 3000, 4096]
    rows = [np.round(rng.standard_normal(max(L, 1)) * 8).astype(np.float32) for L in lens]  # many ties
    return lens, rows


def _rank(rank, world, port, k, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lens, rows = _rows(7)
    width = 4096 // world
    lo = rank * width
    T = len(lens)
    vals = np.zeros((T, k), np.float32)
    idx = np.full((T, k), -1, np.int32)
    for t, L in enumerate(lens):
        n = int(np.clip(L - lo, 0, width))
        sel = oracle.topk(rows[t][lo:lo + n], n, k) if n > 0 else np.full(k, -1, np.int32)
        ok = sel >= 0
        idx[t][ok] = sel[ok] + lo
        vals[t][ok] = rows[t][lo:lo + n][sel[ok]]
    gv = [torch.zeros((T, k), dtype=torch.float32) for _ in range(world)]
    gi = [torch.zeros((T, k), dtype=torch.int32) for _ in range(world)]
    dist.all_gather(gv, torch.from_numpy(vals))
    dist.all_gather(gi, torch.from_numpy(idx))
    merged = []
    for t in range(T):
        cv = np.concatenate([g[t].numpy() for g in gv])
        ci = np.concatenate([g[t].numpy() for g in gi])
        keep = ci >= 0
        cv, ci = cv[keep], ci[keep]  # in rank order, hence in position order
        if len(cv) == 0:
            merged.append(np.full(k, -1, np.int32))
            continue
        slots = oracle.topk(cv, len(cv), k)
        merged.append(np.where(slots >= 0, ci[np.maximum(slots, 0)], -1).astype(np.int32))
    out.put((rank, np.stack(merged)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_merge_to_the_whole_row_selection():
    sys.path.insert(0, ROOT)
    import oracle
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    k = 512
    procs = [ctx.Process(target=_rank, args=(r, 2, port, k, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    lens, rows = _rows(7)
    want = np.stack([oracle.topk(rows[t], L, k) if L > 0 else np.full(k, -1, np.int32) for t, L in enumerate(lens)])
    for rank, got in res:
        assert np.array_equal(got, want), rank
