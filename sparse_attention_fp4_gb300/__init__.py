"""GB300-native FP4 indexer (DeepSeek-V4 sparse-attention index path).

The compute path lives in the CUDA library ``libfp4idx.so`` (C ABI declared in
``include/fp4idx.h``); ``sparse_attention_fp4_gb300.fp4idx`` is its thin Python
binding.  ``workloads`` draws the seeded synthetic inputs.
"""
__all__ = ["workloads"]
