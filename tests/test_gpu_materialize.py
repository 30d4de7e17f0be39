"""Materialised compact workspace (KAP paper, compiler and fallback) through the C ABI.

The cycle copies each view row's selected pages into its request's workspace pages and points the view there. The
proposals must then match the oracle exactly as the zero-copy cycle does (and equal it bit for bit), the workspace
must hold the selected pages byte for byte, the rewritten rows must match the oracle's materialisation, and rows
that do not fit must stay unchanged and flag their request.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PAGE = 16

CASES = [
    dict(name="llama", scale=1 / 16),                     # per-head views
    dict(name="long", scale=1 / 32),                      # one view shared by all heads (span selection)
    dict(name="mixed", scale=1 / 32, ragged=True),        # ragged prompts, per-request A/R/K
    dict(name="mixed", scale=1 / 32, ragged=True, ws=6),  # a workspace smaller than some selections: fallback
    dict(name="llama", scale=1 / 16, ragged=True, unfused=True),  # appends through the full table, then attention
]


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_materialized_cycle(kap, case):
    import oracle
    from tests.gpu_helpers import assert_close_attn, i32, run_cycle_and_oracle
    from workloads import make_workload
    kw = {k: v for k, v in case.items() if k not in ("ws", "unfused")}
    fused = not case.get("unfused", False)
    w = make_workload(device="cuda", **kw)
    ws = case.get("ws") or w.sel_cap()
    res = run_cycle_and_oracle(w, ws_pages=ws, fused=fused)
    cyc = res["cycle"]
    assert np.array_equal(res["nsel_gpu"], res["nsel_orc"])
    for st in res["prop"]:
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, "propose")
    v = res["ver"]
    assert_close_attn(v["o_gpu"], v["o_orc"], v["lse_gpu"], v["lse_orc"], w.dtype, "verify")

    # the view rows, the workspace contents and the fallback flags
    K0 = res["K_pool"][: w.num_pages]
    Kp, Vp = res["K_pool"], res["V_pool"]
    w2 = make_workload(device="cuda", **kw)  # unmodified pool for the byte comparison
    bt = i32(w.block_table)
    vbt, vlp = i32(cyc.view.block_table), i32(cyc.view.logical_page)
    vn, vns = i32(cyc.view.n_entries), i32(cyc.view.n_selected)
    flag = i32(cyc.fallback)
    any_overflow = False
    for r in range(w.R):
        base = w.num_pages + r * ws
        overflow = False
        for row in range(cyc.rows):
            n, ns = int(vn[r, row]), int(vns[r, row])
            orig = np.array([bt[r, lp] for lp in vlp[r, row, :n]], np.int32)
            want, pairs, fits = oracle.materialize_row(orig, vlp[r, row, :n], n, ns, int(w.ctx_len[r]), base, ws)
            assert np.array_equal(vbt[r, row, :n], want), (r, row)
            overflow |= not fits
            heads = [row] if cyc.rows > 1 else list(range(w.Hkv))
            for src, dst in pairs:
                for h in heads:   # bit patterns: unused slots of a partial page hold NaN on both sides
                    assert torch.equal(_bits(Kp[dst, h]), _bits(w2.K[src, h]))
                    assert torch.equal(_bits(Vp[dst, h]), _bits(w2.V[src, h]))
        assert int(flag[r]) == int(overflow), r
        any_overflow |= overflow
    assert any_overflow == ("ws" in case)
    assert kap.kap_device_error() == 0

    # bit for bit the zero-copy cycle on the same inputs
    res0 = run_cycle_and_oracle(w2, fused=fused)
    for i in range(w.k_prop):
        assert torch.equal(_bits(res0["cycle"].o_prop[i]), _bits(cyc.o_prop[i])), i
        assert torch.equal(_bits(res0["cycle"].lse_prop[i]), _bits(cyc.lse_prop[i])), i
    del K0
