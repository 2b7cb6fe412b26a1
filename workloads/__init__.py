"""Seeded synthetic decode workloads (shared by tests, the benchmark and the smoke check).

This module generates inputs only: it holds none of the method's arithmetic
(no scoring, selection, sampling or attention).  See ``synthetic.py``.
"""
from .synthetic import CONFIGS, WorkloadConfig, generate, make_config, budget_split, to_paged

__all__ = ["CONFIGS", "WorkloadConfig", "generate", "make_config", "budget_split", "to_paged"]
