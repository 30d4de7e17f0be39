"""Parity at the benchmark's full sizes and launch configuration: every output checked against the oracle.

At these sizes each CTA of the proposal kernel streams more entries than its ring has slots, so every slot is
reused, and the mixed batch puts more row segments in a CTA's range than one window holds. The oracle still
finishes each case in seconds, so the comparison covers every element, not a sample. Each case runs on its own
and its results are dropped before the next one.
"""
import pytest

pytestmark = pytest.mark.gpu

BIG = [
    dict(name="llama"),                                  # the benchmark workload: 4 x 32768 tokens, A1R2K125
    dict(name="llama", unfused=True),
    dict(name="long"),                                   # 131072 tokens, 451-page span view, 8 proposals
    dict(name="early", batch=8),                         # 8 x 40960 tokens, A0R0K8 per KV head on a noisy proxy
    dict(name="mixed", scale=1 / 4),                     # 32 requests, 1K-32K tokens, many short rows per CTA
]


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


@pytest.mark.parametrize("case", BIG, ids=_id)
def test_full_size_cycle(kap, case):
    import torch
    import tests.test_gpu_parity as tp
    from tests.gpu_helpers import run_cycle_and_oracle
    from workloads import make_workload
    kw = {k: v for k, v in case.items() if k != "unfused"}
    w = make_workload(device="cuda", **kw)
    res = run_cycle_and_oracle(w, fused=not case.get("unfused", False), nthreads=16)
    one = {tp._id(case): (w, res)}
    tp.test_summaries_bit_exact(one, case)
    tp.test_selection_bit_exact(one, case)
    tp.test_view_and_slots_bit_exact(one, case)
    tp.test_append_rope(one, case)
    tp.test_propose_parity(one, case)
    tp.test_verify_parity(one, case)
    assert kap.kap_device_error() == 0
    del one, res, w
    torch.cuda.empty_cache()
