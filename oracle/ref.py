"""ctypes front end of the C oracle (test infrastructure only).

Array conventions match the library's layouts:
  K cache   payload [P,4,64,16] u8, scale [P,4,64] u8
  query     q_payload [T,4,H,16] u8, q_scale [T,4,H] u8
  FP8 cache pages [P, 64*128 + 64*4] u8
bf16 inputs are uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32

PAGE_TOKENS = 64
HEAD_DIM = 128
FP8_PAGE_BYTES = 64 * 128 + 64 * 4


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        sig = {
            "ref_set_threads": (None, [ctypes.c_int]),
            "ref_max_threads": (ctypes.c_int, []),
            "ref_rmsnorm": (None, [_f32p, _f32p, ctypes.c_float, _f32p]),
            "ref_rope": (None, [_f32p, _u16p]),
            "ref_hadamard128": (None, [_f32p]),
            "ref_ue8m0_exponent": (ctypes.c_int, [ctypes.c_float]),
            "ref_ue8m0_byte": (ctypes.c_int, [ctypes.c_float]),
            "ref_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
            "ref_e2m1_code": (ctypes.c_int, [ctypes.c_float]),
            "ref_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
            "ref_e4m3_code": (ctypes.c_int, [ctypes.c_float]),
            "ref_k_chain": (None, [_u16p, _i32, _u16p, ctypes.c_float, _u16p, ctypes.c_int, _f32p]),
            "ref_q_chain": (None, [_u16p, _i32, _u16p, ctypes.c_int, _f32p]),
            "ref_store_k": (ctypes.c_int, [_u16p, _i64, _i32p, _i32p, _u16p, ctypes.c_float, _u16p, _i32,
                                           _u8p, _u8p, _i64]),
            "ref_store_k_fp8": (ctypes.c_int, [_u16p, _i64, _i32p, _i32p, _u16p, ctypes.c_float, _u16p, _i32,
                                               _u8p, _i64]),
            "ref_quant_q": (ctypes.c_int, [_u16p, _i64, _i32, _i32p, _u16p, _i32, _u8p, _u8p]),
            "ref_dequant_k_token": (None, [_u8p, _u8p, _i64, _i32, _f64p]),
            "ref_dequant_q": (None, [_u8p, _u8p, _i32, _i64, _i32, _f64p]),
            "ref_quant_q_fp8": (ctypes.c_int, [_u16p, _i64, _i32, _i32p, _u16p, _i32, _u8p, _f32p]),
            "ref_dequant_k_fp8_token": (None, [_u8p, _i64, _i32, _f64p]),
            "ref_dequant_q_fp8": (None, [_u8p, _f32p, _i32, _i64, _i32, _f64p]),
            "ref_logits_fp8": (ctypes.c_int, [_u8p, _f32p, _f32p, _i64, _i32, _u8p, _i64, _i32p, _i32, _i32p,
                                              _i32p, _i64p, _i64, _i64, _f64p, _f64p]),
            "ref_logits": (ctypes.c_int, [_u8p, _u8p, _f32p, _i64, _i32, _u8p, _u8p, _i64, _i32p, _i32,
                                          _i32p, _i32p, _i64p, _i64, _i64, _f64p, _f64p]),
            "ref_topk": (ctypes.c_int, [_f64p, _i64, _i32, _i32p]),
            "ref_e2m1_codes": (None, [_f32p, _i64, _u8p]),
            "ref_e4m3_codes": (None, [_f32p, _i64, _u8p]),
            "ref_ue8m0_bytes": (None, [_f32p, _i64, _i32p]),
            "ref_fp4_encode_rows": (None, [_f32p, _i64, _u8p, _u8p]),
            "ref_fp4_decode_rows": (None, [_u8p, _u8p, _i64, _f64p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    lib().ref_set_threads(int(n))


def max_threads() -> int:
    return int(lib().ref_max_threads())


# ------------------------------------------------------------------ scalar / element pins
def e2m1_codes(v) -> np.ndarray:
    v = _c(v, np.float32).ravel()
    out = np.empty(v.shape[0], np.uint8)
    lib().ref_e2m1_codes(_p(v, _f32p), v.shape[0], _p(out, _u8p))
    return out


def e2m1_value(code: int) -> float:
    return float(lib().ref_e2m1_value(int(code)))


def e4m3_codes(v) -> np.ndarray:
    v = _c(v, np.float32).ravel()
    out = np.empty(v.shape[0], np.uint8)
    lib().ref_e4m3_codes(_p(v, _f32p), v.shape[0], _p(out, _u8p))
    return out


def e4m3_value(code: int) -> float:
    return float(lib().ref_e4m3_value(int(code)))


def ue8m0_bytes(amax) -> np.ndarray:
    a = _c(amax, np.float32).ravel()
    out = np.empty(a.shape[0], np.int32)
    lib().ref_ue8m0_bytes(_p(a, _f32p), a.shape[0], _p(out, _i32p))
    return out


def rmsnorm(x, w, eps) -> np.ndarray:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    y = np.empty(HEAD_DIM, np.float32)
    lib().ref_rmsnorm(_p(x, _f32p), _p(w, _f32p), float(eps), _p(y, _f32p))
    return y


def rope(u, cos_sin_row) -> np.ndarray:
    u = _c(u, np.float32).copy()
    cs = _c(cos_sin_row, np.uint16)
    lib().ref_rope(_p(u, _f32p), _p(cs, _u16p))
    return u


def hadamard128(u) -> np.ndarray:
    u = _c(u, np.float32).copy()
    lib().ref_hadamard128(_p(u, _f32p))
    return u


def k_chain(k_row, pos, norm_w, eps, cos_sin, stage=3) -> np.ndarray:
    k_row = _c(k_row, np.uint16)
    norm_w = _c(norm_w, np.uint16)
    cos_sin = _c(cos_sin, np.uint16)
    out = np.empty(HEAD_DIM, np.float32)
    lib().ref_k_chain(_p(k_row, _u16p), int(pos), _p(norm_w, _u16p), float(eps), _p(cos_sin, _u16p),
                      int(stage), _p(out, _f32p))
    return out


def q_chain(q_row, pos, cos_sin, stage=3) -> np.ndarray:
    q_row = _c(q_row, np.uint16)
    cos_sin = _c(cos_sin, np.uint16)
    out = np.empty(HEAD_DIM, np.float32)
    lib().ref_q_chain(_p(q_row, _u16p), int(pos), _p(cos_sin, _u16p), int(stage), _p(out, _f32p))
    return out


def fp4_encode_rows(z):
    z = _c(z, np.float32).reshape(-1, HEAD_DIM)
    n = z.shape[0]
    pk = np.empty((n, 4, 16), np.uint8)
    sc = np.empty((n, 4), np.uint8)
    lib().ref_fp4_encode_rows(_p(z, _f32p), n, _p(pk, _u8p), _p(sc, _u8p))
    return pk, sc


def fp4_decode_rows(pk, sc) -> np.ndarray:
    pk = _c(pk, np.uint8).reshape(-1, 4, 16)
    sc = _c(sc, np.uint8).reshape(-1, 4)
    n = pk.shape[0]
    out = np.empty((n, HEAD_DIM), np.float64)
    lib().ref_fp4_decode_rows(_p(pk, _u8p), _p(sc, _u8p), n, _p(out, _f64p))
    return out


# ------------------------------------------------------------------ the path's steps
def store_k(ks, cos_sin, payload=None, scale=None):
    """K store into a split cache; returns (payload, scale, status)."""
    P = int(ks.num_pages)
    if payload is None:
        payload = np.zeros((P, 4, PAGE_TOKENS, 16), np.uint8)
    if scale is None:
        scale = np.zeros((P, 4, PAGE_TOKENS), np.uint8)
    k = _c(ks.k_rows, np.uint16)
    pos = _c(ks.positions, np.int32)
    slots = _c(ks.slots, np.int32)
    nw = _c(ks.norm_w, np.uint16)
    cs = _c(cos_sin, np.uint16)
    st = lib().ref_store_k(_p(k, _u16p), k.shape[0], _p(pos, _i32p), _p(slots, _i32p), _p(nw, _u16p),
                           float(ks.eps), _p(cs, _u16p), cs.shape[0], _p(payload, _u8p), _p(scale, _u8p), P)
    return payload, scale, int(st)


def store_k_fp8(ks, cos_sin, pages=None):
    P = int(ks.num_pages)
    if pages is None:
        pages = np.zeros((P, FP8_PAGE_BYTES), np.uint8)
    k = _c(ks.k_rows, np.uint16)
    pos = _c(ks.positions, np.int32)
    slots = _c(ks.slots, np.int32)
    nw = _c(ks.norm_w, np.uint16)
    cs = _c(cos_sin, np.uint16)
    st = lib().ref_store_k_fp8(_p(k, _u16p), k.shape[0], _p(pos, _i32p), _p(slots, _i32p), _p(nw, _u16p),
                               float(ks.eps), _p(cs, _u16p), cs.shape[0], _p(pages, _u8p), P)
    return pages, int(st)


def quant_q(q, q_positions, cos_sin):
    q = _c(q, np.uint16)
    T, H, Dd = q.shape
    assert Dd == HEAD_DIM
    pos = _c(q_positions, np.int32)
    cs = _c(cos_sin, np.uint16)
    qp = np.zeros((T, 4, H, 16), np.uint8)
    qs = np.zeros((T, 4, H), np.uint8)
    st = lib().ref_quant_q(_p(q, _u16p), T, H, _p(pos, _i32p), _p(cs, _u16p), cs.shape[0], _p(qp, _u8p),
                           _p(qs, _u8p))
    return qp, qs, int(st)


def dequant_k_token(payload, scale, page, j) -> np.ndarray:
    out = np.empty(HEAD_DIM, np.float64)
    payload = _c(payload, np.uint8)
    scale = _c(scale, np.uint8)
    lib().ref_dequant_k_token(_p(payload, _u8p), _p(scale, _u8p), int(page), int(j), _p(out, _f64p))
    return out


def dequant_q(q_payload, q_scale, t, h) -> np.ndarray:
    q_payload = _c(q_payload, np.uint8)
    q_scale = _c(q_scale, np.uint8)
    H = q_payload.shape[2]
    out = np.empty(HEAD_DIM, np.float64)
    lib().ref_dequant_q(_p(q_payload, _u8p), _p(q_scale, _u8p), H, int(t), int(h), _p(out, _f64p))
    return out


def logits(q_payload, q_scale, w, payload, scale, page_table, row_seq, context_lens, rows=None,
           with_bound=True):
    """Binary64 logits for the requested rows: (logits [n, Lmax], bound [n, Lmax] or None, status).
    Entries at s >= L_t are NaN."""
    qp = _c(q_payload, np.uint8)
    qs = _c(q_scale, np.uint8)
    w = _c(w, np.float32)
    pl = _c(payload, np.uint8)
    sc = _c(scale, np.uint8)
    pt = _c(page_table, np.int32)
    rs = _c(row_seq, np.int32)
    cl = _c(context_lens, np.int32)
    T, _, H, _ = qp.shape
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    rows = _c(rows, np.int64)
    Lmax = int(max(1, cl[rows].max() if rows.size else 1))
    out = np.full((rows.shape[0], Lmax), np.nan, np.float64)
    bnd = np.full((rows.shape[0], Lmax), np.nan, np.float64) if with_bound else None
    st = lib().ref_logits(_p(qp, _u8p), _p(qs, _u8p), _p(w, _f32p), T, H, _p(pl, _u8p), _p(sc, _u8p),
                          pl.shape[0], _p(pt, _i32p), pt.shape[1], _p(rs, _i32p), _p(cl, _i32p),
                          _p(rows, _i64p), rows.shape[0], Lmax, _p(out, _f64p),
                          _p(bnd, _f64p) if bnd is not None else None)
    return out, bnd, int(st)


def quant_q_fp8(q, q_positions, cos_sin):
    """FP8 query pack: (q8 [T,8,H,16] u8, q8_scale [T,H] f32, status); the K side's FP8 rule
    per (row, head) after RoPE and the Hadamard."""
    q = _c(q, np.uint16)
    T, H, Dd = q.shape
    assert Dd == HEAD_DIM
    pos = _c(q_positions, np.int32)
    cs = _c(cos_sin, np.uint16)
    q8 = np.zeros((T, 8, H, 16), np.uint8)
    s8 = np.zeros((T, H), np.float32)
    st = lib().ref_quant_q_fp8(_p(q, _u16p), T, H, _p(pos, _i32p), _p(cs, _u16p), cs.shape[0], _p(q8, _u8p),
                               _p(s8, _f32p))
    return q8, s8, int(st)


def dequant_k_fp8_token(pages, page, j) -> np.ndarray:
    out = np.empty(HEAD_DIM, np.float64)
    pages = _c(pages, np.uint8)
    lib().ref_dequant_k_fp8_token(_p(pages, _u8p), int(page), int(j), _p(out, _f64p))
    return out


def dequant_q_fp8(q8, q8_scale, t, h) -> np.ndarray:
    q8 = _c(q8, np.uint8)
    s8 = _c(q8_scale, np.float32)
    out = np.empty(HEAD_DIM, np.float64)
    lib().ref_dequant_q_fp8(_p(q8, _u8p), _p(s8, _f32p), q8.shape[2], int(t), int(h), _p(out, _f64p))
    return out


def logits_fp8(q8, q8_scale, w, pages, page_table, row_seq, context_lens, rows=None, with_bound=True):
    """Binary64 logits over the FP8 operands (the 132 B/token pages of store_k_fp8 and the FP8
    query pack): (logits [n, Lmax], bound or None, status); NaN at s >= L_t."""
    q8 = _c(q8, np.uint8)
    s8 = _c(q8_scale, np.float32)
    w = _c(w, np.float32)
    pg = _c(pages, np.uint8)
    pt = _c(page_table, np.int32)
    rs = _c(row_seq, np.int32)
    cl = _c(context_lens, np.int32)
    T, _, H, _ = q8.shape
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    rows = _c(rows, np.int64)
    Lmax = int(max(1, cl[rows].max() if rows.size else 1))
    out = np.full((rows.shape[0], Lmax), np.nan, np.float64)
    bnd = np.full((rows.shape[0], Lmax), np.nan, np.float64) if with_bound else None
    st = lib().ref_logits_fp8(_p(q8, _u8p), _p(s8, _f32p), _p(w, _f32p), T, H, _p(pg, _u8p), pg.shape[0],
                              _p(pt, _i32p), pt.shape[1], _p(rs, _i32p), _p(cl, _i32p), _p(rows, _i64p),
                              rows.shape[0], Lmax, _p(out, _f64p), _p(bnd, _f64p) if bnd is not None else None)
    return out, bnd, int(st)


def topk(logit_row, L, k) -> np.ndarray:
    lr = _c(logit_row[:L], np.float64)
    out = np.empty(int(k), np.int32)
    st = lib().ref_topk(_p(lr, _f64p), int(L), int(k), _p(out, _i32p))
    assert st == 0
    return out


# ------------------------------------------------------------------ a whole batch
def run_indexer(batch, cos_sin, rows=None):
    """Oracle for one batch: K cache fill, Q quant, logits and top-k of the given rows."""
    payload, scale, st = store_k(batch.kstore, cos_sin)
    assert st == 0
    qp, qs, st = quant_q(batch.q, batch.q_positions, cos_sin)
    assert st == 0
    if rows is None:
        rows = np.arange(batch.n_rows)
    lg, bnd, st = logits(qp, qs, batch.w, payload, scale, batch.page_table, batch.row_seq,
                         batch.context_lens, rows)
    assert st == 0
    tk = np.stack([topk(lg[i], int(batch.context_lens[r]), batch.topk) for i, r in enumerate(rows)]) \
        if len(rows) else np.zeros((0, batch.topk), np.int32)
    return dict(payload=payload, scale=scale, q_payload=qp, q_scale=qs, logits=lg, bound=bnd,
                topk=tk, rows=np.asarray(rows))


# ------------------------------------------------------------------ head weights
def bf16_values(bits) -> np.ndarray:
    """bf16 bit patterns -> their exact values in binary64 (a bf16 is the top half of a
    float32)."""
    b = np.ascontiguousarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def head_weights(hidden, w_proj, w_scale):
    """[P1] Summary ("a one-launch index-Q pack + head weights"; indexer_head_weights runs a
    bf16 GEMV whose result stays in fp32): w[t,h] = w_scale * sum_d hidden[t,d] *
    w_proj[h,d] in binary64 (bf16 products are exact there), and the bound
    |w_scale| * sum_d |hidden[t,d] * w_proj[h,d]| that device rounding is measured against.
    hidden [T, D] and w_proj [H, D] are bf16 bit patterns; w_scale is taken as an fp32."""
    h = bf16_values(hidden)
    w = bf16_values(w_proj)
    s = float(np.float32(w_scale))
    return s * (h @ w.T), abs(s) * (np.abs(h) @ np.abs(w).T)
