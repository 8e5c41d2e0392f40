"""Helpers for the GPU parity tests: move the seeded numpy inputs to the device."""
import numpy as np
import torch


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype) if t.element_size() == torch.empty(0, dtype=dtype).element_size() else t.to(dtype)
    return t.cuda()


def bf16(a):
    """uint16 bf16 bit patterns -> torch.bfloat16 CUDA tensor (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    return t.detach().cpu().numpy()


def kstore_to_device(ks):
    return dict(k=bf16(ks.k_rows), positions=dev(ks.positions), slots=dev(ks.slots), norm_w=bf16(ks.norm_w))


def run_gpu_indexer(b, cos_sin_np, with_logits=True, page_table=None, payload=None, scale=None, k=None,
                    fused=False):
    """Whole path on the GPU through the binding: K store, Q quant, schedule, logits + top-k
    (fp4idx_logits_topk, or fp4idx_logits_topk_fused with fused=True)."""
    from sparse_attention_fp4_gb300 import fp4idx
    cs = bf16(cos_sin_np)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if payload is None:
        ks = b.kstore
        payload, scale = fp4idx.alloc_cache(b.num_pages)
        fp4idx.store_k(bf16(ks.k_rows), dev(ks.positions), dev(ks.slots), bf16(ks.norm_w), ks.eps, cs, payload,
                       scale, status=status)
    T = b.n_rows
    k = b.topk if k is None else k
    qp, qs = fp4idx.alloc_query(T)
    fp4idx.quant_q(bf16(b.q), dev(b.q_positions), cs, qp, qs, status=status)
    cl, rs = dev(b.context_lens), dev(b.row_seq)
    Lmax = int(max(1, b.context_lens.max()))
    sched = torch.empty(fp4idx.schedule_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    fp4idx.build_schedule(cl, rs, sched)
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    pt = dev(b.page_table if page_table is None else page_table)
    ws = torch.empty(fp4idx.logits_workspace_bytes(T, Lmax, k), dtype=torch.uint8, device="cuda")
    if with_logits:
        lg = torch.full((T, Lmax), float("nan"), dtype=torch.float32, device="cuda")
    else:
        lg = None
    fp4idx.logits_topk(qp, qs, dev(b.w), payload, scale, pt, rs, cl, Lmax, k, sched, ws, topk, logits_out=lg,
                       status=status, fused=fused)
    torch.cuda.synchronize()
    return dict(status=fp4idx.read_status(status), payload=payload, scale=scale, q_payload=qp, q_scale=qs,
                logits=None if lg is None else lg.cpu().numpy(), topk=topk.cpu().numpy())


def check_logits(got_row, ref_row, bound_row, L, what=""):
    err = np.abs(got_row[:L].astype(np.float64) - ref_row[:L])
    tol = 1e-5 * bound_row[:L] + 1e-6
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, "%s logits: %d of %d outside tolerance, first s=%d gpu=%r oracle=%r tol=%r" % (
        what, bad.size, L, bad[0], got_row[bad[0]], ref_row[bad[0]], tol[bad[0]])


def check_topk(got, ref_row, bound_row, L, k, what=""):
    """Selection = k highest oracle logits up to swaps among values within tolerance of the
    k-th; ascending positions; -1 padding."""
    sel = got[got >= 0]
    m = min(L, k)
    assert sel.size == m, "%s: %d selected, expected %d" % (what, sel.size, m)
    assert np.all(got[m:] == -1) and np.all(got[:m] >= 0), what
    assert np.all(np.diff(sel) > 0) and (sel.size == 0 or sel.max() < L), what
    if L <= k:
        assert np.array_equal(sel, np.arange(L)), what
        return
    lr = ref_row[:L]
    tol = 1e-5 * bound_row[:L] + 1e-6
    order = np.lexsort((np.arange(L), -lr))
    ref_set = set(order[:k].tolist())
    thresh = lr[order[k - 1]]
    t_tol = tol[order[k - 1]]
    got_set = set(sel.tolist())
    for s in got_set - ref_set:
        assert lr[s] >= thresh - tol[s] - t_tol, "%s: token %d (%r) selected below the k-th %r" % (what, s, lr[s], thresh)
    for s in ref_set - got_set:
        assert lr[s] <= thresh + tol[s] + t_tol, "%s: token %d (%r) dropped above the k-th %r" % (what, s, lr[s], thresh)


def check_topk_self(got, lg_row, L, k, what=""):
    """The selection is exactly the top-k of the kernel's own logits (index tie-break)."""
    order = np.lexsort((np.arange(L), -lg_row[:L].astype(np.float64)))
    exp = np.sort(order[:min(L, k)])
    assert np.array_equal(got[got >= 0], exp), what
