"""Host-side argument validation of the C ABI, on CPU: every entry point rejects null
pointers, misaligned buffers, bad sizes and unsupported shapes with the status code
include/fp4idx.h documents, before it touches the GPU (each case here fails validation,
so nothing is launched), and the size queries return 0 for impossible requests."""
import ctypes

import pytest

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 4
V = ctypes.c_void_p
I64, I32, F32, SZ = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
A = V(1 << 20)   # a 16-byte aligned address (never dereferenced: validation fails first)
M4 = V((1 << 20) + 4)  # 4-byte but not 16-byte aligned
M1 = V((1 << 20) + 1)  # not even 4-byte aligned


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_fp4_gb300 import build
    L = ctypes.CDLL(build.build())
    sig = {
        "fp4idx_store_k": [V, I64, V, V, V, F32, V, I32, V, V, I64, V, V],
        "fp4idx_quant_q": [V, I64, I32, V, V, I32, V, V, V, V],
        "fp4idx_quant_q_w": [V, I64, I32, V, V, I32, V, I32, V, F32, V, V, V, V, V],
        "fp4idx_build_schedule": [V, V, I64, I32, V, SZ, V],
        "fp4idx_prepare_step": [V, I64, V, V, V, F32, V, I64, I32, V, V, I32, V, V, I64, V, V, V, V, I32, V, SZ, V, V],
        "fp4idx_topk": [V, I64, V, I64, I32, I32, V, SZ, V, V, V],
        "fp4idx_topk_noalloc": [V, I64, V, I64, I32, I32, V, V, V],
        "fp4idx_topk_values": [V, I64, V, I64, I32, V, V],
        "fp4idx_topk_merge": [V, V, I64, I32, I32, V, SZ, V, V, V],
        "fp4idx_dequant_pages": [V, V, I64, V, I64, V, V, V],
        "fp4idx_export_pages": [V, V, I64, V, I64, V, V, V, V],
        "fp4idx_import_pages": [V, V, V, I64, V, V, I64, V, V],
        "fp4idx_logits_fp8": [V, V, V, I64, I32, V, I64, V, I64, I32, V, V, I32, V, SZ, V, I64, V, V],
        "fp4idx_logits_topk_fp8": [V, V, V, I64, I32, V, I64, V, I64, I32, V, V, I32, I32, V, SZ, V, SZ, V, V, I64,
                                   V, V],
        "fp4idx_read_status": [V, V, V],
    }
    for name, args in sig.items():
        getattr(L, name).argtypes = args
        getattr(L, name).restype = ctypes.c_int
    for name, args in {"fp4idx_schedule_workspace_bytes": [I64, I32],
                       "fp4idx_topk_workspace_bytes": [I64, I32],
                       "fp4idx_logits_workspace_bytes": [I64, I32, I32],
                       "fp4idx_topk_merge_workspace_bytes": [I64, I32, I32]}.items():
        getattr(L, name).argtypes = args
        getattr(L, name).restype = SZ
    L.fp4idx_status_string.restype = ctypes.c_char_p
    return L


def test_store_k(lib):
    f = lib.fp4idx_store_k
    assert f(A, -1, A, A, A, 1e-6, A, 16, A, A, 8, None, None) == INVALID
    assert f(A, 0, None, None, None, 1e-6, None, 16, None, None, 8, None, None) == OK  # nothing to do
    assert f(A, 4, None, A, A, 1e-6, A, 16, A, A, 8, None, None) == INVALID          # null positions
    assert f(M4, 4, A, A, A, 1e-6, A, 16, A, A, 8, None, None) == INVALID            # k misaligned
    assert f(A, 4, A, A, A, 1e-6, A, 0, A, A, 8, None, None) == INVALID              # empty RoPE table
    assert f(A, 4, A, A, A, 1e-6, A, 16, A, A, 1 << 26, None, None) == UNSUPPORTED   # slots overflow int32


def test_quant_q_and_quant_q_w(lib):
    q = lib.fp4idx_quant_q
    assert q(A, 1, 32, A, A, 16, A, A, None, None) == UNSUPPORTED                  # heads != 64
    assert q(A, 1, 64, A, A, 16, None, A, None, None) == INVALID
    assert q(A, 0, 64, None, None, 16, None, None, None, None) == OK
    qw = lib.fp4idx_quant_q_w
    args = lambda T, H, D, w_out=A, hidden=A: (A, T, H, A, A, 16, hidden, D, A, 1.0, A, A, w_out, None, None)
    assert qw(*args(1, 64, 100)) == UNSUPPORTED        # hidden size not a multiple of 256
    assert qw(*args(1, 64, 16384 + 256)) == UNSUPPORTED
    assert qw(*args(1, 32, 256)) == UNSUPPORTED
    assert qw(*args(1, 64, 256, w_out=None)) == INVALID
    assert qw(*args(1, 64, 256, hidden=M4)) == INVALID
    assert qw(*args(-1, 64, 256)) == INVALID


def test_schedule(lib):
    f = lib.fp4idx_build_schedule
    assert f(A, A, -1, 152, A, 1 << 20, None) == INVALID
    assert f(A, A, 4, 152, None, 1 << 20, None) == INVALID
    assert f(A, A, 4, 152, M4, 1 << 20, None) == INVALID
    assert f(None, A, 4, 152, A, 1 << 20, None) == INVALID
    need = lib.fp4idx_schedule_workspace_bytes(4, 152)
    assert need > 0 and f(A, A, 4, 152, A, need - 1, None) == WORKSPACE
    assert lib.fp4idx_schedule_workspace_bytes(-1, 152) == 0


def test_prepare_step(lib):
    f = lib.fp4idx_prepare_step
    def args(**kw):
        a = dict(k=A, n_new=4, pos=A, slots=A, norm_w=A, eps=1e-6, q=A, n_rows=2, heads=64, qpos=A, cs=A, max_pos=16,
                 payload=A, scale=A, num_pages=8, qp=A, qs=A, cl=A, rs=A, num_ctas=152, sched=A, sched_bytes=1 << 20,
                 status=None)
        a.update(kw)
        return (a["k"], a["n_new"], a["pos"], a["slots"], a["norm_w"], a["eps"], a["q"], a["n_rows"], a["heads"],
                a["qpos"], a["cs"], a["max_pos"], a["payload"], a["scale"], a["num_pages"], a["qp"], a["qs"], a["cl"],
                a["rs"], a["num_ctas"], a["sched"], a["sched_bytes"], a["status"], None)
    assert f(*args(n_new=-1)) == INVALID
    assert f(*args(heads=32)) == UNSUPPORTED
    assert f(*args(pos=None)) == INVALID          # K store arguments
    assert f(*args(payload=M4)) == INVALID
    assert f(*args(q=None)) == INVALID            # Q quant arguments
    assert f(*args(qp=M4)) == INVALID
    assert f(*args(cl=M1)) == INVALID             # schedule arguments
    assert f(*args(sched=None)) == INVALID
    assert f(*args(sched=M4)) == INVALID
    assert f(*args(status=M1)) == INVALID
    need = lib.fp4idx_schedule_workspace_bytes(2, 152)
    assert f(*args(sched_bytes=need - 1)) == WORKSPACE
    assert f(*args(max_pos=0)) == INVALID


def test_topk(lib):
    f = lib.fp4idx_topk
    assert f(A, 100, A, 2, 100, 0, A, 1 << 20, A, None, None) == INVALID            # k = 0
    assert f(A, 100, A, 2, 100, 4097, A, 1 << 20, A, None, None) == INVALID         # k above the maximum
    assert f(A, 70000, A, 2, 70000, 16, A, 1 << 30, A, None, None) == UNSUPPORTED   # context above the maximum
    assert f(A, 50, A, 2, 100, 16, A, 1 << 20, A, None, None) == INVALID            # stride below max_context
    assert f(M1, 100, A, 2, 100, 16, A, 1 << 20, A, None, None) == INVALID
    assert f(A, 100, A, 2, 100, 16, A, 0, A, None, None) == WORKSPACE
    assert lib.fp4idx_topk_workspace_bytes(-1, 100) == 0


def test_topk_noalloc(lib):
    """Argument errors are reported before the fixed scratch's set-up (a CUDA call) runs."""
    SCRATCH_LIMIT = 10
    f = lib.fp4idx_topk_noalloc
    assert f(A, 100, A, 2, 100, 0, A, None, None) == INVALID             # k = 0
    assert f(A, 100, A, 2, 100, 4097, A, None, None) == INVALID          # k above the maximum
    assert f(A, 100, A, -1, 100, 16, A, None, None) == INVALID           # negative rows
    assert f(A, 70000, A, 2, 70000, 16, A, None, None) == UNSUPPORTED    # context above the maximum
    assert f(None, 100, A, 2, 100, 16, A, None, None) == INVALID         # null logits
    assert f(A, 100, None, 2, 100, 16, A, None, None) == INVALID         # null context_lens
    assert f(A, 100, A, 2, 100, 16, None, None, None) == INVALID         # null output
    assert f(M1, 100, A, 2, 100, 16, A, None, None) == INVALID           # logits misaligned
    assert f(A, 100, M1, 2, 100, 16, A, None, None) == INVALID
    assert f(A, 100, A, 2, 100, 16, M1, None, None) == INVALID
    assert f(A, 100, A, 2, 100, 16, A, M1, None) == INVALID              # status misaligned
    assert f(A, 50, A, 2, 100, 16, A, None, None) == INVALID             # stride below max_context
    # 128 rows of 65,536 fit the 16 MiB exactly; one more row does not
    assert lib.fp4idx_topk_workspace_bytes(128, 65536) <= 16 << 20
    assert f(A, 65536, A, 129, 65536, 16, A, None, None) == SCRATCH_LIMIT
    assert f(None, 65536, None, 129, 65536, 16, None, None, None) == SCRATCH_LIMIT


def test_topk_values_and_merge(lib):
    v = lib.fp4idx_topk_values
    assert v(A, 100, A, 2, 0, A, None) == INVALID
    assert v(A, 0, A, 2, 16, A, None) == INVALID
    assert v(None, 100, A, 2, 16, A, None) == INVALID
    m = lib.fp4idx_topk_merge
    assert m(A, A, 2, 4, 0, A, 1 << 30, A, None, None) == INVALID                   # k = 0
    assert m(A, A, 2, 40, 2048, A, 1 << 30, A, None, None) == INVALID               # shards * k too large
    assert m(A, A, 2, 2000, 16, A, 1 << 30, A, None, None) == INVALID               # too many shards
    assert m(A, A, 2, 4, 16, M4, 1 << 30, A, None, None) == INVALID                 # workspace misaligned
    need = lib.fp4idx_topk_merge_workspace_bytes(2, 4, 16)
    assert need > 0 and m(A, A, 2, 4, 16, A, need - 1, A, None, None) == WORKSPACE
    assert lib.fp4idx_topk_merge_workspace_bytes(2, 40, 2048) == 0
    assert m(None, None, 0, 4, 16, None, 0, None, None, None) == OK                 # no rows


def test_pages(lib):
    d = lib.fp4idx_dequant_pages
    assert d(A, A, -1, A, 1, A, None, None) == INVALID
    assert d(A, A, 10, None, 1, A, None, None) == INVALID
    assert d(A, A, 10, A, 1, M4, None, None) == INVALID
    assert d(None, None, 10, None, 0, None, None, None) == OK
    e = lib.fp4idx_export_pages
    assert e(A, A, 10, A, -1, A, A, None, None) == INVALID
    assert e(A, M4, 10, A, 1, A, A, None, None) == INVALID
    assert e(A, A, 10, M1, 1, A, A, None, None) == INVALID
    i = lib.fp4idx_import_pages
    assert i(A, A, A, 1, A, A, -1, None, None) == INVALID
    assert i(None, A, A, 1, A, A, 10, None, None) == INVALID


def test_status_strings(lib):
    names = [lib.fp4idx_status_string(c).decode() for c in range(11)]
    assert len(set(names)) == 11 and "unknown status" not in names
    assert lib.fp4idx_status_string(99).decode() == "unknown status"
    assert lib.fp4idx_read_status(None, None, None) == INVALID


def test_logits_fp8(lib):
    f = lib.fp4idx_logits_fp8

    def call(q8=A, s8=A, w=A, n=4, heads=64, pages=A, P=8, pt=A, rs=A, cl=A, max_ctx=256, sched=A, status=None):
        return f(q8, s8, w, n, heads, pages, P, pt, 2, 4, rs, cl, max_ctx, sched, 1 << 20, A, 256, status, None)

    assert call(n=-1) == INVALID
    assert call(heads=32) == UNSUPPORTED
    assert call(max_ctx=(1 << 30)) == UNSUPPORTED
    assert call(n=0, q8=None, pages=None) == OK  # nothing to do
    assert call(q8=None) == INVALID
    assert call(pages=None) == INVALID
    assert call(s8=M4) == INVALID      # q8_scale must be 16-byte aligned
    assert call(pages=M4) == INVALID   # the tensor map wants a 16-byte aligned base
    assert call(cl=M1) == INVALID
    assert call(status=M1) == INVALID


def test_logits_topk_fp8(lib):
    f = lib.fp4idx_logits_topk_fp8

    def call(q8=A, s8=A, n=4, heads=64, pages=A, max_ctx=256, k=16, status=None):
        return f(q8, s8, A, n, heads, pages, 8, A, 2, 4, A, A, max_ctx, k, A, 1 << 20, A, 1 << 24, A, None, 0,
                 status, None)

    assert call(n=-1) == INVALID
    assert call(heads=128) == UNSUPPORTED
    assert call(max_ctx=(1 << 30)) == UNSUPPORTED
    assert call(q8=None) == INVALID
    assert call(s8=M4) == INVALID
    assert call(pages=M1) == INVALID
    assert call(status=M1) == INVALID
