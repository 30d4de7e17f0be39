"""Seeded synthetic inputs for the selected-KV decode hot path.

This module only draws random numbers and lays them out (KV pools, block tables, queries, spans, per-request
policies). It holds none of the method's arithmetic: no summary, score, selection, view, RoPE or attention.
Both the CUDA library's tests/bench and the CPU oracle take their inputs from here.
"""
from .gen import Workload, make_workload, make_prior, make_verify_logits, CONFIGS  # noqa: F401
