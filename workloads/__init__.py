"""Seeded synthetic workloads for paged-KV attention (inputs only)."""
from .configs import CONFIGS, BENCH_CONFIG
from .gen import Case, PrefillPart, make_case, empty_cache, rope_cos_sin

__all__ = ["CONFIGS", "BENCH_CONFIG", "Case", "PrefillPart", "make_case", "empty_cache"]
