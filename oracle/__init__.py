"""CPU oracle for the FP4 indexer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``fp4idx_ref.c`` (plain C, built
with ``-ffp-contract=off``) through ctypes and adds numpy conveniences.  It shares
no code with the CUDA library and never imports the product package except its
input generators (``sparse_attention_fp4_gb300.workloads``), which hold none of
the method's arithmetic.
"""
from .ref import *  # noqa: F401,F403
