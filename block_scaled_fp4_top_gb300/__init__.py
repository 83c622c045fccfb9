"""GB300-native routed MoE FFN layer with block-scaled FP4 (NVFP4) experts.

The compute lives in ``libfp4moe.so`` (CUDA for sm_103a, C ABI in
``include/fp4moe.h``). ``block_scaled_fp4_top_gb300.api`` is the thin torch
binding. Importing this package loads nothing. The library is loaded on the
first API call, and that call raises if the library has not been built.
"""

__all__ = ["api", "build"]
