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


def test_mixed_serving_batch_at_full_size(kap):
    """The mixed serving batch at its stated size: 32 requests with prompts log-uniform in 4K-128K tokens, per-request
    retention s in {2, 5.5, 10, 25}% and splits A1R2 / A4R4 / A0R0, one proposal launch for every request and one
    verify launch with windows of 2, 4 or 8, all pages scattered over a shared 2^20-page pool (64 GiB of K and V).
    The oracle runs request by request on that request's own pages; every element is compared."""
    import numpy as np
    import torch
    from tests.gpu_helpers import LSE_TOL, TOL, assert_close_attn, run_cycle_per_request
    from workloads import make_workload
    w = make_workload("mixed", device="cuda")
    assert w.num_pages == 1 << 20 and w.R == 32
    ctx = w.ctx_len.cpu().numpy()
    assert ctx.min() >= 4096 and ctx.max() < 131072
    seen = 0
    for res in run_cycle_per_request(w, nthreads=16):
        r = res["r"]
        assert np.array_equal(res["S_gpu"].view(np.uint32), res["S_orc"].view(np.uint32)), r
        assert np.array_equal(res["scores_gpu"].view(np.uint32), res["scores_orc"].view(np.uint32)), r
        assert np.array_equal(res["nsel_gpu"], res["nsel_orc"]), r
        for v in range(len(res["nsel_orc"])):
            n = res["nsel_orc"][v]
            assert np.array_equal(res["sel_gpu"][v, :n], res["sel_orc"][v, :n]), (r, v)
        for (cbt, clog, ns), (gbt, glp, gns) in res["view"]:
            assert gns == ns and np.array_equal(gbt, cbt) and np.array_equal(glp, clog), r
        for g_slot, o_slot in res["slots"]:
            assert g_slot == o_slot, r
        Kg, Ko = res["K_after"]
        Vg, Vo = res["V_after"]
        assert np.array_equal(np.isnan(Kg), np.isnan(Ko)) and np.array_equal(np.isnan(Vg), np.isnan(Vo)), r
        m = ~np.isnan(Ko)
        ulp = np.maximum(np.abs(Ko[m]), 1e-30) * 2.0 ** -7
        assert (np.abs(Kg[m] - Ko[m]) <= 2 * ulp + 2.0 ** -19 * res["k_in_max"]).all(), r
        assert np.array_equal(Vg[~np.isnan(Vo)], Vo[~np.isnan(Vo)]), r
        for i, (og, oo, lg, lo) in enumerate(res["prop"]):
            assert_close_attn(og, oo, lg, lo, w.dtype, f"request {r} proposal {i}")
        og, oo, lg, lo = res["ver"]
        assert_close_attn(og, oo, lg, lo, w.dtype, f"request {r} verify")
        seen += 1
    assert seen == 32
    assert kap.kap_device_error() == 0
    del w
    torch.cuda.empty_cache()
