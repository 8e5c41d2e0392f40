"""Python binding of libfp4idx.so (C ABI in include/fp4idx.h).

Argument marshalling only: every step of the indexer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors on the current device; bf16 data may be
passed as torch.bfloat16 or as int16/uint16 bit patterns.  Calls enqueue work on
the current torch stream (or the stream given) and return immediately.  If the
library has not been built, importing this module raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4idx.so")

HEAD_DIM = 128
NUM_HEADS = 64
PAGE_TOKENS = 64
FP8_PAGE_BYTES = 64 * 128 + 64 * 4
MAX_TOPK = 4096
MAX_CONTEXT = 65536

STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error", 4: "workspace too small",
    5: "page id or slot outside the cache", 6: "pipeline wait timed out", 7: "RoPE position outside the table",
    8: "context length out of range", 9: "schedule does not match the call",
    10: "call needs more than the fixed top-k scratch",
}


class Fp4IdxError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (status %d)" % (fn, STATUS.get(code, "unknown"), code))
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError("libfp4idx.so is not built (expected at %s); run __graft_entry__.build() or "
                      "python -m sparse_attention_fp4_gb300.build" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "fp4idx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp4idx_num_sms": (ctypes.c_int, [ctypes.POINTER(_i32)]),
    "fp4idx_store_k": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp, _f32, _vp, _i32, _vp, _vp, _i64, _vp, _vp]),
    "fp4idx_store_k_fp8": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp, _f32, _vp, _i32, _vp, _i64, _vp, _vp]),
    "fp4idx_quant_q": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "fp4idx_quant_q_fp8": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "fp4idx_quant_q_w": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _f32, _vp, _vp, _vp, _vp,
                                        _vp]),
    "fp4idx_prepare_step": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp, _f32, _vp, _i64, _i32, _vp, _vp, _i32, _vp, _vp,
                                           _i64, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp, _vp]),
    "fp4idx_schedule_workspace_bytes": (_sz, [_i64, _i32]),
    "fp4idx_build_schedule": (ctypes.c_int, [_vp, _vp, _i64, _i32, _vp, _sz, _vp]),
    "fp4idx_logits_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "fp4idx_logits_topk": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _vp, _vp, _i64, _vp, _i64, _i32, _vp, _vp,
                                          _i32, _i32, _vp, _sz, _vp, _sz, _vp, _vp, _i64, _vp, _vp]),
    "fp4idx_logits_topk_fused": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _vp, _vp, _i64, _vp, _i64, _i32, _vp,
                                                _vp, _i32, _i32, _vp, _sz, _vp, _sz, _vp, _vp, _i64, _vp, _vp]),
    "fp4idx_logits": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _vp, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _i32,
                                     _vp, _sz, _vp, _i64, _vp, _vp]),
    "fp4idx_logits_fp8": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _i32,
                                         _vp, _sz, _vp, _i64, _vp, _vp]),
    "fp4idx_logits_topk_fp8": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _vp, _i64, _vp, _i64, _i32, _vp, _vp, _i32,
                                              _i32, _vp, _sz, _vp, _sz, _vp, _vp, _i64, _vp, _vp]),
    "fp4idx_topk_workspace_bytes": (_sz, [_i64, _i32]),
    "fp4idx_topk": (ctypes.c_int, [_vp, _i64, _vp, _i64, _i32, _i32, _vp, _sz, _vp, _vp, _vp]),
    "fp4idx_topk_noalloc": (ctypes.c_int, [_vp, _i64, _vp, _i64, _i32, _i32, _vp, _vp, _vp]),
    "fp4idx_dequant_pages": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _vp, _vp]),
    "fp4idx_export_pages": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp]),
    "fp4idx_import_pages": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "fp4idx_topk_merge_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "fp4idx_topk_values": (ctypes.c_int, [_vp, _i64, _vp, _i64, _i32, _vp, _vp]),
    "fp4idx_topk_merge": (ctypes.c_int, [_vp, _vp, _i64, _i32, _i32, _vp, _sz, _vp, _vp, _vp]),
    "fp4idx_test_pipeline_waits": (ctypes.c_int, [_i32, _i64]),
    "fp4idx_read_status": (ctypes.c_int, [_vp, ctypes.POINTER(_i32), _vp]),
}

EXPORTS = tuple(_SIGS)

for _name, (_res, _args) in _SIGS.items():
    if hasattr(_lib, _name):
        _fn = getattr(_lib, _name)
        _fn.restype = _res
        _fn.argtypes = _args


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t, name, dtypes=None, numel=None, nullable=False):
    if t is None:
        if nullable:
            return None
        raise ValueError("%s is required" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if numel is not None and t.numel() < numel:
        raise ValueError("%s has %d elements, needs %d" % (name, t.numel(), numel))
    return ctypes.c_void_p(t.data_ptr())


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_U8 = (torch.uint8,)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def _check(fn, rc):
    if rc != 0:
        raise Fp4IdxError(fn, rc)


def num_sms() -> int:
    n = _i32(0)
    _check("fp4idx_num_sms", _lib.fp4idx_num_sms(ctypes.byref(n)))
    return int(n.value)


# ------------------------------------------------------------------ cache / query allocation helpers
def alloc_cache(num_pages, device="cuda"):
    """Split FP4 cache: (payload [P,4,64,16] u8, scale [P,4,64] u8), zeroed."""
    return (torch.zeros((num_pages, 4, PAGE_TOKENS, 16), dtype=torch.uint8, device=device),
            torch.zeros((num_pages, 4, PAGE_TOKENS), dtype=torch.uint8, device=device))


def alloc_query(n_rows, device="cuda"):
    return (torch.empty((n_rows, 4, NUM_HEADS, 16), dtype=torch.uint8, device=device),
            torch.empty((n_rows, 4, NUM_HEADS), dtype=torch.uint8, device=device))


# ------------------------------------------------------------------ entry points
def store_k(k, positions, slots, norm_w, eps, cos_sin, payload, scale, status=None, stream=None):
    n = k.shape[0] if k.dim() == 2 else 0
    if k.dim() != 2 or k.shape[1] != HEAD_DIM:
        raise ValueError("k must be [n_rows, 128]")
    num_pages = payload.shape[0]
    rc = _lib.fp4idx_store_k(
        _ptr(k, "k", _BF16), n, _ptr(positions, "positions", _I32, n), _ptr(slots, "slots", _I32, n),
        _ptr(norm_w, "norm_w", _BF16, HEAD_DIM), float(eps), _ptr(cos_sin, "cos_sin", _BF16), cos_sin.shape[0],
        _ptr(payload, "payload", _U8, num_pages * 4096), _ptr(scale, "scale", _U8, num_pages * 256), num_pages,
        _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_store_k", rc)


def store_k_fp8(k, positions, slots, norm_w, eps, cos_sin, pages, status=None, stream=None):
    n = k.shape[0]
    if k.dim() != 2 or k.shape[1] != HEAD_DIM:
        raise ValueError("k must be [n_rows, 128]")
    num_pages = pages.shape[0]
    rc = _lib.fp4idx_store_k_fp8(
        _ptr(k, "k", _BF16), n, _ptr(positions, "positions", _I32, n), _ptr(slots, "slots", _I32, n),
        _ptr(norm_w, "norm_w", _BF16, HEAD_DIM), float(eps), _ptr(cos_sin, "cos_sin", _BF16), cos_sin.shape[0],
        _ptr(pages, "pages", _U8, num_pages * FP8_PAGE_BYTES), num_pages,
        _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_store_k_fp8", rc)


def quant_q(q, q_positions, cos_sin, q_payload, q_scale, status=None, stream=None):
    if q.dim() != 3 or q.shape[2] != HEAD_DIM:
        raise ValueError("q must be [n_rows, heads, 128]")
    T, H = q.shape[0], q.shape[1]
    rc = _lib.fp4idx_quant_q(
        _ptr(q, "q", _BF16), T, H, _ptr(q_positions, "q_positions", _I32, T), _ptr(cos_sin, "cos_sin", _BF16),
        cos_sin.shape[0], _ptr(q_payload, "q_payload", _U8, T * 4096), _ptr(q_scale, "q_scale", _U8, T * 256),
        _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_quant_q", rc)


def quant_q_fp8(q, q_positions, cos_sin, q8, q8_scale, status=None, stream=None):
    """FP8 query pack: q8 [T, 8, 64, 16] uint8 and q8_scale [T, 64] fp32."""
    T, H, D = q.shape
    rc = _lib.fp4idx_quant_q_fp8(_ptr(q, "q", _BF16, T * H * D), T, H, _ptr(q_positions, "q_positions", _I32, T),
                                 _ptr(cos_sin, "cos_sin", _BF16), cos_sin.shape[0], _ptr(q8, "q8", _U8, T * 8192),
                                 _ptr(q8_scale, "q8_scale", _F32, T * NUM_HEADS),
                                 _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_quant_q_fp8", rc)


def quant_q_w(q, q_positions, cos_sin, hidden, w_proj, w_scale, q_payload, q_scale, w_out, status=None,
              stream=None):
    """fp4idx_quant_q and the head weights w_out = w_scale * hidden @ w_proj^T in one launch."""
    T, H, D = q.shape
    dim = hidden.shape[1]
    rc = _lib.fp4idx_quant_q_w(_ptr(q, "q", _BF16, T * H * D), T, H, _ptr(q_positions, "q_positions", _I32, T),
                               _ptr(cos_sin, "cos_sin", _BF16), cos_sin.shape[0],
                               _ptr(hidden, "hidden", _BF16, T * dim), dim, _ptr(w_proj, "w_proj", _BF16, NUM_HEADS * dim),
                               float(w_scale), _ptr(q_payload, "q_payload", _U8, T * 4096),
                               _ptr(q_scale, "q_scale", _U8, T * 256), _ptr(w_out, "w_out", _F32, T * NUM_HEADS),
                               _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_quant_q_w", rc)


def schedule_workspace_bytes(max_rows, num_ctas=0) -> int:
    return int(_lib.fp4idx_schedule_workspace_bytes(int(max_rows), int(num_ctas)))


def logits_workspace_bytes(max_rows, max_context, k) -> int:
    return int(_lib.fp4idx_logits_workspace_bytes(int(max_rows), int(max_context), int(k)))


def build_schedule(context_lens, row_seq, schedule, num_ctas=0, stream=None):
    T = context_lens.numel()
    rc = _lib.fp4idx_build_schedule(
        _ptr(context_lens, "context_lens", _I32, T), _ptr(row_seq, "row_seq", _I32, T), T, int(num_ctas),
        _ptr(schedule, "schedule", _U8), schedule.numel(), _stream_ptr(stream))
    _check("fp4idx_build_schedule", rc)


def prepare_step(k, positions, slots, norm_w, eps, q, q_positions, cos_sin, payload, scale, q_payload, q_scale,
                 context_lens, row_seq, schedule, num_ctas=0, status=None, stream=None):
    """fp4idx_prepare_step: the K store of the new rows, the Q quant and the schedule build
    in one launch (the results of store_k, quant_q and build_schedule)."""
    n_new = k.shape[0]
    if k.dim() != 2 or k.shape[1] != HEAD_DIM:
        raise ValueError("k must be [n_new, 128]")
    if q.dim() != 3 or q.shape[2] != HEAD_DIM:
        raise ValueError("q must be [n_rows, heads, 128]")
    T, H = q.shape[0], q.shape[1]
    num_pages = payload.shape[0]
    rc = _lib.fp4idx_prepare_step(
        _ptr(k, "k", _BF16, nullable=n_new == 0), n_new, _ptr(positions, "positions", _I32, n_new, nullable=n_new == 0),
        _ptr(slots, "slots", _I32, n_new, nullable=n_new == 0), _ptr(norm_w, "norm_w", _BF16, HEAD_DIM), float(eps),
        _ptr(q, "q", _BF16), T, H, _ptr(q_positions, "q_positions", _I32, T), _ptr(cos_sin, "cos_sin", _BF16),
        cos_sin.shape[0], _ptr(payload, "payload", _U8, num_pages * 4096), _ptr(scale, "scale", _U8, num_pages * 256),
        num_pages, _ptr(q_payload, "q_payload", _U8, T * 4096), _ptr(q_scale, "q_scale", _U8, T * 256),
        _ptr(context_lens, "context_lens", _I32, T), _ptr(row_seq, "row_seq", _I32, T), int(num_ctas),
        _ptr(schedule, "schedule", _U8), schedule.numel(), _ptr(status, "status", _I32, 1, nullable=True),
        _stream_ptr(stream))
    _check("fp4idx_prepare_step", rc)


def logits_topk(q_payload, q_scale, w, payload, scale, page_table, row_seq, context_lens, max_context, k,
                schedule, workspace, topk_idx, logits_out=None, status=None, stream=None, fused=False):
    """fp4idx_logits_topk (the logits launch, then the top-k launch), or with fused=True
    fp4idx_logits_topk_fused (the selection inside the logits launch; writes `schedule`)."""
    T = q_payload.shape[0]
    num_pages = payload.shape[0]
    S, max_pages = page_table.shape
    stride = logits_out.shape[1] if logits_out is not None else 0
    fn = _lib.fp4idx_logits_topk_fused if fused else _lib.fp4idx_logits_topk
    rc = fn(
        _ptr(q_payload, "q_payload", _U8, T * 4096), _ptr(q_scale, "q_scale", _U8, T * 256),
        _ptr(w, "w", _F32, T * NUM_HEADS), T, NUM_HEADS, _ptr(payload, "payload", _U8, num_pages * 4096),
        _ptr(scale, "scale", _U8, num_pages * 256), num_pages, _ptr(page_table, "page_table", _I32), S, max_pages,
        _ptr(row_seq, "row_seq", _I32, T), _ptr(context_lens, "context_lens", _I32, T), int(max_context), int(k),
        _ptr(schedule, "schedule", _U8), schedule.numel(),
        _ptr(workspace, "workspace", _U8), workspace.numel(),
        _ptr(topk_idx, "topk_idx", _I32, T * int(k)), _ptr(logits_out, "logits_out", _F32, nullable=True),
        stride, _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_logits_topk_fused" if fused else "fp4idx_logits_topk", rc)


def logits(q_payload, q_scale, w, payload, scale, page_table, row_seq, context_lens, max_context, schedule,
           logits_out, status=None, stream=None):
    T = q_payload.shape[0]
    num_pages = payload.shape[0]
    S, max_pages = page_table.shape
    rc = _lib.fp4idx_logits(
        _ptr(q_payload, "q_payload", _U8, T * 4096), _ptr(q_scale, "q_scale", _U8, T * 256),
        _ptr(w, "w", _F32, T * NUM_HEADS), T, NUM_HEADS, _ptr(payload, "payload", _U8, num_pages * 4096),
        _ptr(scale, "scale", _U8, num_pages * 256), num_pages, _ptr(page_table, "page_table", _I32), S, max_pages,
        _ptr(row_seq, "row_seq", _I32, T), _ptr(context_lens, "context_lens", _I32, T), int(max_context),
        _ptr(schedule, "schedule", _U8), schedule.numel(), _ptr(logits_out, "logits_out", _F32),
        logits_out.shape[1], _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_logits", rc)


def logits_fp8(q8, q8_scale, w, fp8_pages, page_table, row_seq, context_lens, max_context, schedule, logits_out,
               status=None, stream=None):
    """Paged-MQA logits over the FP8 comparison cache (fp8_pages [P, 8448] u8) and the FP8
    query pack (q8 [T, 8, 64, 16] u8, q8_scale [T, 64] f32)."""
    T = q8.shape[0]
    num_pages = fp8_pages.shape[0]
    S, max_pages = page_table.shape
    rc = _lib.fp4idx_logits_fp8(
        _ptr(q8, "q8", _U8, T * 8192), _ptr(q8_scale, "q8_scale", _F32, T * NUM_HEADS),
        _ptr(w, "w", _F32, T * NUM_HEADS), T, NUM_HEADS, _ptr(fp8_pages, "fp8_pages", _U8, num_pages * FP8_PAGE_BYTES),
        num_pages, _ptr(page_table, "page_table", _I32), S, max_pages, _ptr(row_seq, "row_seq", _I32, T),
        _ptr(context_lens, "context_lens", _I32, T), int(max_context), _ptr(schedule, "schedule", _U8),
        schedule.numel(), _ptr(logits_out, "logits_out", _F32), logits_out.shape[1],
        _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_logits_fp8", rc)


def logits_topk_fp8(q8, q8_scale, w, fp8_pages, page_table, row_seq, context_lens, max_context, k, schedule,
                    workspace, topk_idx, logits_out=None, status=None, stream=None):
    """FP8 logits and the top-k selection in one call (workspace: logits_workspace_bytes)."""
    T = q8.shape[0]
    num_pages = fp8_pages.shape[0]
    S, max_pages = page_table.shape
    stride = logits_out.shape[1] if logits_out is not None else 0
    rc = _lib.fp4idx_logits_topk_fp8(
        _ptr(q8, "q8", _U8, T * 8192), _ptr(q8_scale, "q8_scale", _F32, T * NUM_HEADS),
        _ptr(w, "w", _F32, T * NUM_HEADS), T, NUM_HEADS, _ptr(fp8_pages, "fp8_pages", _U8, num_pages * FP8_PAGE_BYTES),
        num_pages, _ptr(page_table, "page_table", _I32), S, max_pages, _ptr(row_seq, "row_seq", _I32, T),
        _ptr(context_lens, "context_lens", _I32, T), int(max_context), int(k), _ptr(schedule, "schedule", _U8),
        schedule.numel(), _ptr(workspace, "workspace", _U8), workspace.numel(),
        _ptr(topk_idx, "topk_idx", _I32, T * int(k)), _ptr(logits_out, "logits_out", _F32, nullable=True), stride,
        _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_logits_topk_fp8", rc)


def topk_workspace_bytes(max_rows, max_context) -> int:
    return int(_lib.fp4idx_topk_workspace_bytes(int(max_rows), int(max_context)))


def topk(logits_buf, context_lens, max_context, k, workspace, topk_idx, status=None, stream=None):
    T = context_lens.numel()
    rc = _lib.fp4idx_topk(_ptr(logits_buf, "logits", _F32), logits_buf.shape[1],
                          _ptr(context_lens, "context_lens", _I32, T), T, int(max_context), int(k),
                          _ptr(workspace, "workspace", _U8), workspace.numel(),
                          _ptr(topk_idx, "topk_idx", _I32, T * int(k)), _ptr(status, "status", _I32, 1, nullable=True),
                          _stream_ptr(stream))
    _check("fp4idx_topk", rc)


TOPK_NOALLOC_MAX_BYTES = 16 * 1024 * 1024  # FP4IDX_TOPK_NOALLOC_MAX_BYTES


def topk_noalloc(logits_buf, context_lens, max_context, k, topk_idx, status=None, stream=None):
    """fp4idx_topk with the library's fixed per-device scratch: no workspace argument."""
    T = context_lens.numel()
    rc = _lib.fp4idx_topk_noalloc(_ptr(logits_buf, "logits", _F32), logits_buf.shape[1],
                                  _ptr(context_lens, "context_lens", _I32, T), T, int(max_context), int(k),
                                  _ptr(topk_idx, "topk_idx", _I32, T * int(k)),
                                  _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_topk_noalloc", rc)


def dequant_pages(payload, scale, page_ids, out, status=None, stream=None):
    """out[i] = the fp32 values of page page_ids[i] of the split cache ([n, 64, 128])."""
    n = page_ids.numel()
    num_pages = payload.shape[0]
    rc = _lib.fp4idx_dequant_pages(_ptr(payload, "payload", _U8, num_pages * 4096),
                                   _ptr(scale, "scale", _U8, num_pages * 256), num_pages,
                                   _ptr(page_ids, "page_ids", _I32, n), n, _ptr(out, "out", _F32, n * 64 * 128),
                                   _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_dequant_pages", rc)


def export_pages(payload, scale, page_ids, rows_payload, rows_scale, status=None, stream=None):
    """Page rows of the listed pages: rows_payload [n, 4096] and rows_scale [n, 256] uint8."""
    n = page_ids.numel()
    num_pages = payload.shape[0]
    rc = _lib.fp4idx_export_pages(_ptr(payload, "payload", _U8, num_pages * 4096),
                                  _ptr(scale, "scale", _U8, num_pages * 256), num_pages,
                                  _ptr(page_ids, "page_ids", _I32, n), n,
                                  _ptr(rows_payload, "rows_payload", _U8, n * 4096),
                                  _ptr(rows_scale, "rows_scale", _U8, n * 256),
                                  _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_export_pages", rc)


def import_pages(rows_payload, rows_scale, page_ids, payload, scale, status=None, stream=None):
    """Writes page page_ids[i] of the split cache from page row i (ids distinct)."""
    n = page_ids.numel()
    num_pages = payload.shape[0]
    rc = _lib.fp4idx_import_pages(_ptr(rows_payload, "rows_payload", _U8, n * 4096),
                                  _ptr(rows_scale, "rows_scale", _U8, n * 256), _ptr(page_ids, "page_ids", _I32, n),
                                  n, _ptr(payload, "payload", _U8, num_pages * 4096),
                                  _ptr(scale, "scale", _U8, num_pages * 256), num_pages,
                                  _ptr(status, "status", _I32, 1, nullable=True), _stream_ptr(stream))
    _check("fp4idx_import_pages", rc)


def topk_values(logits_buf, topk_idx, values, stream=None):
    """values[t][i] = logits_buf[t][topk_idx[t][i]] (-inf for -1 padding)."""
    T, k = topk_idx.shape
    rc = _lib.fp4idx_topk_values(_ptr(logits_buf, "logits", _F32), logits_buf.shape[1],
                                 _ptr(topk_idx, "topk_idx", _I32, T * k), T, k, _ptr(values, "values", _F32, T * k),
                                 _stream_ptr(stream))
    _check("fp4idx_topk_values", rc)


def topk_merge_workspace_bytes(max_rows, n_shards, k) -> int:
    return int(_lib.fp4idx_topk_merge_workspace_bytes(int(max_rows), int(n_shards), int(k)))


def topk_merge(cand_values, cand_idx, workspace, topk_idx, status=None, stream=None):
    """Row top-k from per-shard candidates [T, n_shards, k] (global positions, shards in
    position order)."""
    T, S, k = cand_idx.shape
    rc = _lib.fp4idx_topk_merge(_ptr(cand_values, "cand_values", _F32, T * S * k),
                                _ptr(cand_idx, "cand_idx", _I32, T * S * k), T, S, k,
                                _ptr(workspace, "workspace", _U8), workspace.numel(),
                                _ptr(topk_idx, "topk_idx", _I32, T * k), _ptr(status, "status", _I32, 1, nullable=True),
                                _stream_ptr(stream))
    _check("fp4idx_topk_merge", rc)


def test_pipeline_waits(idle_producers: bool, wait_limit_ns: int = 0) -> None:
    """Test switch of the logits kernels' bounded waits: with idle_producers the producer
    warps of later logits launches issue nothing, so every wait runs out after
    wait_limit_ns and the launch records FP4IDX_ERR_TIMEOUT.  (False, 0) restores normal
    operation and the default limit."""
    _check("fp4idx_test_pipeline_waits", _lib.fp4idx_test_pipeline_waits(1 if idle_producers else 0,
                                                                          int(wait_limit_ns)))


def read_status(status, stream=None) -> int:
    out = _i32(0)
    _check("fp4idx_read_status", _lib.fp4idx_read_status(_ptr(status, "status", _I32, 1), ctypes.byref(out),
                                                        _stream_ptr(stream)))
    return int(out.value)
