"""Standalone measurements of the memory-system floors behind the attention
kernels' design (TMA streaming of the K/V tile pattern from HBM and from L2,
the latency of reading split states other CTAs have just written). Not part of
the library: they build their own executable.

    python -m gqa_kv_head_gb300.probes
"""
