"""Plain fp64 CPU oracle for the decode-attention hot path.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
benchmark's CPU-baseline / reference arm may import this package. The product
path (include/fr_kernels.h, gqa_kv_head_gb300/) never imports, links or calls
it, and it shares no code with the CUDA kernels.
"""
from .fr_oracle import (yarn_corr_dims, rope_theta, rope_theta_f32, rope_theta_scale_f32, rope_neox, qkv_post, kv_append,
                        attention_collapsed, attention_batched, attention_rows,
                        attention_split_merge, split_partials, merge_partials,
                        decode_attn, f16_round)

__all__ = ["yarn_corr_dims", "rope_theta", "rope_theta_f32", "rope_theta_scale_f32", "rope_neox", "qkv_post", "kv_append",
           "attention_collapsed", "attention_batched", "attention_rows",
           "attention_split_merge", "split_partials", "merge_partials",
           "decode_attn", "f16_round"]
