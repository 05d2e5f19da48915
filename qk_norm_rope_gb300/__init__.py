"""Fused QK-RMSNorm + multi-axis RoPE + scaled-dot-product attention for GB300.

The computation lives in the CUDA library ``libst_rope_attn.so`` (C-ABI in
``include/st_rope_attn.h``); ``qk_norm_rope_gb300.api`` is its ctypes binding.
Importing this package loads nothing; the library is built and loaded on the
first call.
"""
__all__ = ["api", "build"]
