"""GB300-native RocketKV decode hot path: SnapKV++ eviction + Hybrid Sparse Attention.

The compute path is the CUDA library ``librkv.so`` (C-ABI declared in
``include/rkv.h``); ``two_stage_kv_snapkv_gb300.rkv`` is its thin Python binding.
Importing this package does not load the library; importing ``.rkv`` does, and
fails loudly when it has not been built.
"""
__all__ = ["rkv", "workloads"]
