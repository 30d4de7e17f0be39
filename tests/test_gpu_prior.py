"""External-prior selection (KRI page, prior schema) through the C ABI against the oracle.

The prior block_affinities[L][H][N] of each request is mean-pooled over layers and heads in the library's fixed fp32
order, then the A<a>R<r>K<k> top-K is taken per request. Pooled scores and selections must match bit for bit.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PAGE = 16

CASES = [
    dict(name="llama", scale=1 / 16, L=32),                # 256 rows: 8 full chunks
    dict(name="llama", scale=1 / 16, L=5, H=7),            # 35 rows: a partial second chunk
    dict(name="llama", scale=1 / 16, L=32, quantize=0.5),  # coarse values: pooled scores tie, lower page wins
    dict(name="mixed", scale=1 / 32, ragged=True, L=16),   # ragged prompts, per-request A/R/K
    dict(name="llama", scale=1.0, L=32),                   # the full Llama-shaped layer: 4 x 2048 pages
]


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


def _run(kap, c):
    from workloads import make_prior, make_workload
    import oracle
    w = make_workload(c["name"], device="cuda", scale=c["scale"], ragged=c.get("ragged", False), poison=False)
    aff = make_prior(w, c["L"], device="cpu", quantize=c.get("quantize"))
    if "H" in c:  # a prior with its own head count (the connector pools whatever heads the baker wrote)
        aff = torch.randn(aff.shape[0], c["L"], c["H"], aff.shape[3], generator=torch.Generator().manual_seed(5))
    aff_dev = aff.contiguous().to("cuda")
    R, max_pages = w.R, int(w.block_table.shape[1])
    ark = w.ark.cpu()
    same = bool((ark == ark[0]).all())
    a0, r0, k0 = (int(x) for x in ark[0].tolist())
    ctx = w.ctx_len.cpu().numpy()
    N = (ctx + PAGE - 1) // PAGE
    cap = int(max(min(int(n), int(a) + int(rr) + int(k)) for n, (a, rr, k) in zip(N, ark.tolist())))
    pol = kap.AccessPolicy(a0, r0, k0, False, cap, None if same else w.ark.contiguous())
    pmap = kap.PageMap(w.block_table, w.ctx_len)
    sel = torch.full((R, 1, cap), -7, dtype=torch.int32, device="cuda")
    nsel = torch.zeros((R, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(kap.kap_score_workspace_size(R, 1, max_pages) // 4, dtype=torch.float32, device="cuda")
    kap.kap_prior_topk(pmap, aff_dev, pol, sel, nsel, ws)
    torch.cuda.synchronize()
    scores_gpu = ws[: R * max_pages].view(R, max_pages).cpu().numpy()
    sel_gpu, nsel_gpu = sel.cpu().numpy(), nsel.cpu().numpy()
    a_np = aff.numpy()
    for r in range(R):
        n = int(N[r])
        sc = oracle.prior_scores(a_np[r, :, :, :n])
        assert np.array_equal(scores_gpu[r, :n].view(np.uint32), sc.view(np.uint32)), f"scores of request {r}"
        a, rr, k = (int(x) for x in ark[r].tolist())
        ids = oracle.topk_ark(sc, n, a, rr, k)
        assert int(nsel_gpu[r, 0]) == len(ids), f"count of request {r}"
        assert np.array_equal(sel_gpu[r, 0, :len(ids)], np.asarray(ids, np.int32)), f"selection of request {r}"
        if c.get("quantize") is not None:
            assert len(set(sc[a:n - rr].tolist())) < n - a - rr, "the quantised prior should produce tied scores"
        # a prior that favours the needle pages selects them (all of them fit in k)
        if w.needles and w.needles[r] and k >= len(w.needles[r]) and "H" not in c:
            assert set(w.needles[r]) <= set(ids)
    assert kap.kap_device_error() == 0


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_prior_selection_bit_exact(kap, case):
    _run(kap, case)
