"""GB300 (sm_103a) decode-attention hot path for a ggml host: qkv_post (NEOX
RoPE with YaRN, scale, f16 t-major Q rows) and the collapsed GQA decode
attention over one shared f16 KV head, behind the C ABI in include/fr_kernels.h.

The kernels live in csrc/ and build into _build/libfr_gb300.so (build.py).
This Python layer only marshals arguments (ops.py over ctypes, _abi.py).
"""
from ._abi import FR_ROPE_EXACT, FR_ROPE_GGML_F32, FrError, FrRopeParams, library_path, load
from .ops import (decode_attn, decode_attn_noalloc, decode_attn_noalloc_check, decode_attn_plan, kv_append, make_workspace, qkv_post,
                  rope_params,
                  workspace_check, workspace_size)

__all__ = ["FR_ROPE_EXACT", "FR_ROPE_GGML_F32", "FrError", "FrRopeParams", "library_path", "load", "decode_attn", "decode_attn_noalloc",
           "decode_attn_noalloc_check",
           "decode_attn_plan", "kv_append", "make_workspace",
           "qkv_post", "rope_params", "workspace_check", "workspace_size"]
