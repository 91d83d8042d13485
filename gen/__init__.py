"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package holds no arithmetic of the attention method itself: only a
counter-based random generator (rng.py) and the workload recipes (workloads.py)
that turn it into Q, positions, K, V and masks of the documented shapes.
"""
from .rng import uniform, normal, splitmix64_stream
from .workloads import (Workload, RopeParams, make_workload, named_config,
                        NAMED_CONFIGS, SWEEP_HD, SWEEP_NTOK, SWEEP_NKV,
                        sweep_config)

__all__ = ["uniform", "normal", "splitmix64_stream", "Workload", "RopeParams",
           "make_workload", "named_config", "NAMED_CONFIGS", "SWEEP_HD",
           "SWEEP_NTOK", "SWEEP_NKV", "sweep_config"]
