"""The fused entry points against the pairs of calls they replace, on identical inputs.

kap_score_topk_view must produce exactly what kap_score_topk followed by kap_compile_view produces: the selection,
the view and the horizon's slot mapping, compared bit for bit.

kap_append_propose must produce what kap_append_kv (the step token at seq_len-1, q rotated) followed by
kap_attn_propose produces:
- the pool contents after the step, bit for bit;
- the attention outputs and LSEs, to within 1e-6 in fp32 or one bf16 rounding step. The fused kernel rotates q in
  the same arithmetic, but its warps may merge a split row in a different order.

A proposal launch with a settled view (kap_view.settled: scan and prompt-page copies start before the dependency
wait) must produce exactly what the same launch produces when it waits first: only the timing differs.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [dict(name="tiny"), dict(name="llama", scale=1 / 16), dict(name="mixed", scale=1 / 32, ragged=True),
         dict(name="early", scale=1 / 16, batch=3)]


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


def _cycle(kap, w, fused):
    from tests.gpu_helpers import make_cycle
    pool, cyc = make_cycle(w, fused=fused)
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    return pool, cyc


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_score_topk_view_equals_separate_calls(kap, case):
    from workloads import make_workload
    outs = []
    for fused in (True, False):
        w = make_workload(device="cuda", **case)
        _, cyc = _cycle(kap, w, fused)
        cyc.plan(w.q_route)
        torch.cuda.synchronize()
        outs.append({k: getattr(cyc.view, k).cpu().clone() for k in ("block_table", "logical_page", "n_entries",
                                                                     "n_selected")} |
                    {"sel": cyc.sel_ids.cpu().clone(), "nsel": cyc.n_sel.cpu().clone(),
                     "slots": cyc.slots_prop.cpu().clone(), "pos": cyc.pos_prop.cpu().clone(),
                     "fallback": cyc.fallback.cpu().clone()})
    a, b = outs
    for k in ("n_entries", "n_selected", "nsel", "slots", "pos", "fallback"):
        assert torch.equal(a[k], b[k]), k
    R, rows, _ = a["sel"].shape
    for r in range(R):
        for v in range(rows):
            n = int(a["n_entries"][r, v])
            ns = int(a["nsel"][r, v])
            assert torch.equal(a["block_table"][r, v, :n], b["block_table"][r, v, :n])
            assert torch.equal(a["logical_page"][r, v, :n], b["logical_page"][r, v, :n])
            assert torch.equal(a["sel"][r, v, :ns], b["sel"][r, v, :ns])
    assert kap.kap_device_error() == 0


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_append_propose_equals_append_then_propose(kap, case):
    from workloads import make_workload
    res = []
    for fused in (True, False):
        w = make_workload(device="cuda", **case)
        pool, cyc = _cycle(kap, w, fused)
        cyc.plan(w.q_route)
        q = w.q_prop.clone()
        for i in range(w.k_prop):
            cyc.propose_step(i, q[i], w.k_new_prop[i], w.v_new_prop[i])
        torch.cuda.synchronize()
        res.append(dict(o=cyc.o_prop.float().cpu(), lse=cyc.lse_prop.cpu(), K=w.K.cpu(), V=w.V.cpu()))
    f, u = res
    nan_k = torch.isnan(f["K"])
    assert torch.equal(nan_k, torch.isnan(u["K"]))
    assert torch.equal(f["K"][~nan_k], u["K"][~nan_k])
    nan_v = torch.isnan(f["V"])
    assert torch.equal(f["V"][~nan_v], u["V"][~nan_v])
    if f["o"].dtype == torch.float32 and case["name"] == "tiny":
        atol = 1e-6
    else:
        atol = float(np.abs(u["o"].numpy()).max()) * 2.0 ** -7 + 1e-6
    assert torch.allclose(f["o"], u["o"], atol=atol, rtol=0)
    assert torch.allclose(f["lse"], u["lse"], atol=1e-5, rtol=0)
    assert kap.kap_device_error() == 0


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_settled_view_changes_nothing(kap, case, fused):
    from tests.gpu_helpers import make_cycle
    from workloads import make_workload
    res = []
    for overlap in (True, False):
        w = make_workload(device="cuda", **case)
        pool, cyc = make_cycle(w, fused=fused, overlap=overlap)
        kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
        cyc.plan(w.q_route)
        torch.cuda.synchronize()  # the view is complete before the first proposal launch: every step may be settled
        q = w.q_prop.clone()
        for i in range(w.k_prop):
            cyc.propose_step(i, q[i], w.k_new_prop[i], w.v_new_prop[i], settled=True if overlap else None)
        torch.cuda.synchronize()
        res.append(dict(o=cyc.o_prop.cpu(), lse=cyc.lse_prop.cpu(), K=w.K.cpu(), V=w.V.cpu()))
    a, b = res
    for k in ("o", "lse", "K", "V"):
        nan = torch.isnan(a[k])
        assert torch.equal(nan, torch.isnan(b[k])), k
        assert torch.equal(a[k][~nan], b[k][~nan]), k
    assert kap.kap_device_error() == 0
