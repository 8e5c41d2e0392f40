"""The C-ABI library builds, loads and exports every entry point include/fp4idx.h
declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "fp4idx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4idx_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from sparse_attention_fp4_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    names = declared_entry_points()
    assert len(names) >= 10
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from sparse_attention_fp4_gb300 import build
    build.build()
    from sparse_attention_fp4_gb300 import fp4idx
    assert set(declared_entry_points()) <= set(fp4idx.EXPORTS)


def test_host_side_validation_without_gpu():
    """Argument checks run before any CUDA call, so they answer on a machine without a GPU."""
    from sparse_attention_fp4_gb300 import build
    lib = ctypes.CDLL(build.build())
    lib.fp4idx_quant_q.restype = ctypes.c_int
    # heads != 64 -> UNSUPPORTED; negative rows -> INVALID_ARG; null pointers -> INVALID_ARG
    assert lib.fp4idx_quant_q(None, ctypes.c_int64(1), ctypes.c_int32(32), None, None, ctypes.c_int32(10),
                              None, None, None, None) == 2
    assert lib.fp4idx_quant_q(None, ctypes.c_int64(-1), ctypes.c_int32(64), None, None, ctypes.c_int32(10),
                              None, None, None, None) == 1
    assert lib.fp4idx_quant_q(None, ctypes.c_int64(4), ctypes.c_int32(64), None, None, ctypes.c_int32(10),
                              None, None, None, None) == 1
    lib.fp4idx_status_string.restype = ctypes.c_char_p
    assert lib.fp4idx_status_string(5) == b"page id or slot outside the cache"
