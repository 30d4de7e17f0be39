"""Memory-traffic cost model of one proposal/verification cycle (test infrastructure only).

KAP paper, Section 4 (cost model), with the equations as printed in its agifrontier.github.io tutorial:
  Cost_base = (1 + k h) (W_main + KV)                 plain decoding of as many tokens as a cycle yields
  Cost_plan = k (W_prop + s KV) + (W_main + KV)       k selected-KV proposals, then one full verification
  with W_prop = W_main the plan wins iff (h - s) KV > (1 - h) W_main     (Eq. 9, the phase boundary)
  KV_crit = (1 - h) W_main / (h - s)                  the context size at which the boundary is crossed
s is the retained-KV ratio of the proposal path, h the proposal acceptance rate, k the proposal length.
"""
from __future__ import annotations


def cost_base(k: int, h: float, w_main: float, kv: float) -> float:
    return (1.0 + k * h) * (w_main + kv)


def cost_plan(k: int, s: float, w_prop: float, w_main: float, kv: float) -> float:
    return k * (w_prop + s * kv) + (w_main + kv)


def plan_wins(h: float, s: float, w_main: float, kv: float) -> bool:
    """Phase boundary for a self-speculative plan (W_prop = W_main)."""
    return (h - s) * kv > (1.0 - h) * w_main


def kv_crit(h: float, s: float, w_main: float) -> float:
    """Critical KV cost above which the plan pays off; requires h > s."""
    if h <= s:
        return float("inf")
    return (1.0 - h) * w_main / (h - s)


def cycle_kv_bytes(k: int, s: float, kv_bytes: float) -> float:
    """KV bytes one planned cycle reads (Cost_plan with the weight terms set to zero)."""
    return k * s * kv_bytes + kv_bytes
