"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by element, on seeded workloads.

Indices, tables and slots must match bit-exactly; attention outputs within max-abs 2e-2 (bf16 I/O, fp32
accumulation) or 1e-4 (fp32 KV); log-sum-exp within 1e-3.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="tiny"),
    dict(name="tiny", ragged=True),
    dict(name="llama", scale=1 / 16),
    dict(name="llama", scale=1 / 16, ragged=True),
    dict(name="long", scale=1 / 32),
    dict(name="early", scale=1 / 16, batch=3),
    dict(name="mixed", scale=1 / 32),
    dict(name="mixed", scale=1 / 32, ragged=True),
    # 72 short requests: 576 attention rows, more than the proposal kernel scans in shared memory at once
    dict(name="mixed", scale=1 / 64, batch=72, ragged=True),
    dict(name="llama", scale=1 / 32, n_q_override=5),   # verify window k + 1 (carry + 4 candidates)
    dict(name="llama", scale=1 / 32, n_q_override=2),   # window shorter than the proposals: appends stay visible
    dict(name="llama", scale=1 / 32, n_q_override=16),  # G * n_q = 64 query columns: the widest verification tile
    # proposal steps as separate kap_append_kv + kap_attn_propose calls (the others use kap_append_propose)
    dict(name="tiny", unfused=True),
    dict(name="llama", scale=1 / 16, unfused=True),
    dict(name="mixed", scale=1 / 32, ragged=True, unfused=True),
]


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


@pytest.fixture(scope="module")
def results(kap):
    from tests.gpu_helpers import run_cycle_and_oracle
    from workloads import make_workload
    out = {}
    for c in CASES:
        kw = {k: v for k, v in c.items() if k != "unfused"}
        w = make_workload(device="cuda", **kw)
        out[_id(c)] = (w, run_cycle_and_oracle(w, fused=not c.get("unfused", False)))
    return out


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_summaries_bit_exact(results, case):
    w, res = results[_id(case)]
    bt = w.block_table.cpu().numpy()
    ctx = w.ctx_len.cpu().numpy()
    for r in range(w.R):
        N = (int(ctx[r]) + 15) // 16
        pages = bt[r, :N]
        assert np.array_equal(res["S_gpu"][pages], res["S_orc"][pages])


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_selection_bit_exact(results, case):
    w, res = results[_id(case)]
    assert np.array_equal(res["nsel_gpu"], res["nsel_orc"])
    R, rows, _ = res["sel_orc"].shape
    for r in range(R):
        for v in range(rows):
            n = res["nsel_orc"][r, v]
            assert np.array_equal(res["sel_gpu"][r, v, :n], res["sel_orc"][r, v, :n]), (r, v)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_view_and_slots_bit_exact(results, case):
    import oracle
    w, res = results[_id(case)]
    cyc = res["cycle"]
    bt = w.block_table.cpu().numpy()
    ctx, seq0 = w.ctx_len.cpu().numpy(), w.seq_len0.cpu().numpy()
    vbt, vlp = cyc.view.block_table.cpu().numpy(), cyc.view.logical_page.cpu().numpy()
    vn, vns = cyc.view.n_entries.cpu().numpy(), cyc.view.n_selected.cpu().numpy()
    for r in range(w.R):
        for v in range(cyc.rows):
            n = res["nsel_orc"][r, v]
            cbt, clog, nsel = oracle.compile_view_row(bt[r], int(ctx[r]), int(seq0[r]), cyc.horizon,
                                                      res["sel_orc"][r, v, :n])
            assert vn[r, v] == len(cbt) and vns[r, v] == nsel
            assert np.array_equal(vbt[r, v, :len(cbt)], cbt) and np.array_equal(vlp[r, v, :len(clog)], clog)
    slots = cyc.slots_prop.cpu().numpy().reshape(w.R, cyc.horizon)
    pos = cyc.pos_prop.cpu().numpy().reshape(w.R, cyc.horizon)
    for r in range(w.R):
        for i in range(cyc.horizon):
            assert pos[r, i] == seq0[r] + i
            assert slots[r, i] == oracle.slot(bt[r], int(seq0[r]) + i)
    qo = w.q_offsets.cpu().numpy()
    sv = cyc.slots_ver.cpu().numpy()
    pv = cyc.pos_ver.cpu().numpy()
    for r in range(w.R):
        for j in range(qo[r], qo[r + 1]):
            assert pv[j] == seq0[r] + (j - qo[r])
            assert sv[j] == oracle.slot(bt[r], int(pv[j]))


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_scores_bit_exact(results, case):
    """The Q.K page scores themselves (not only the selection they lead to): bit-identical to the oracle's fixed-order
    fp32 scores for every prompt page of every row."""
    w, res = results[_id(case)]
    if "scores_gpu" not in res:
        pytest.skip("span selection has no scores")
    ctx = w.ctx_len.cpu().numpy()
    g, o = res["scores_gpu"], res["scores_orc"]
    for r in range(w.R):
        N = (int(ctx[r]) + 15) // 16
        assert np.array_equal(g[r, :, :N].view(np.uint32), o[r, :, :N].view(np.uint32)), r


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_append_rope(results, case):
    w, res = results[_id(case)]
    Kg, Ko = res["K_after_gpu"], res["K_after_orc"]
    Vg, Vo = res["V_after_gpu"], res["V_after_orc"]
    # every slot the oracle wrote or kept must match; untouched poisoned slots stay NaN on both sides
    assert np.array_equal(np.isnan(Kg), np.isnan(Ko)) and np.array_equal(np.isnan(Vg), np.isnan(Vo))
    m = ~np.isnan(Ko)
    if w.dtype == torch.float32:
        assert np.abs(Kg[m] - Ko[m]).max() <= 1e-5
    else:
        # Two bf16 ulps of the value, plus the fp32 rotation error. The latter scales with the rotated pair's inputs,
        # not with the result, which can cancel to far below them: allow 2^-19 of the largest input key.
        ulp = np.maximum(np.abs(Ko[m]), 1e-30) * 2.0 ** -7
        kin = max(float(w.k_new_prop.abs().max()), float(w.k_new_ver.abs().max()))
        assert (np.abs(Kg[m] - Ko[m]) <= 2 * ulp + 2.0 ** -19 * kin).all()
    assert np.array_equal(Vg[~np.isnan(Vo)], Vo[~np.isnan(Vo)])
    for st in res["prop"]:   # unfused steps rotate the queries in place at their positions
        if st["q_gpu"] is None:
            continue
        tol = 1e-5 if w.dtype == torch.float32 else 2 * 2.0 ** -7
        assert np.abs(st["q_gpu"] - st["q_orc"]).max() <= tol * max(1.0, np.abs(st["q_orc"]).max())


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_propose_parity(results, case):
    from tests.gpu_helpers import assert_close_attn
    w, res = results[_id(case)]
    for i, st in enumerate(res["prop"]):
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, f"propose step {i}")


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_verify_parity(results, case):
    from tests.gpu_helpers import assert_close_attn
    w, res = results[_id(case)]
    v = res["ver"]
    assert_close_attn(v["o_gpu"], v["o_orc"], v["lse_gpu"], v["lse_orc"], w.dtype, "verify")


def test_needles_are_selected(results):
    # sanity (not exactness): pages whose keys were pushed 3 sigma toward the query are routed to
    w, res = results[_id(dict(name="llama", scale=1 / 16))]
    k_mid = int(w.ark[0, 2])
    for r in range(w.R):
        for h in range(w.Hkv):
            chosen = set(res["sel_gpu"][r, h, : res["nsel_gpu"][r, h]].tolist())
            hit = sum(p in chosen for p in w.needles[r])
            assert hit >= min(len(w.needles[r]), k_mid) // 2


def test_no_device_errors(results, kap):
    assert kap.kap_device_error() == 0
