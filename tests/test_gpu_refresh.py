"""Refresh of the K summaries of listed pages (kap_refresh_summaries) after tokens are committed into the prompt.

Each request's prompt first ends a few tokens earlier (the state before a commit); then ctx_len grows to the full
prompt and only the touched pages are refreshed: the page that was partial and the pages that are new. The result
must equal, bit for bit, a full rebuild over the grown prompts and the oracle's block means. Unused slots hold NaN,
so a refresh that read past a page's valid tokens would show.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [("tiny", dict(ragged=True)), ("llama", dict(scale=1 / 16, ragged=True)),
         ("mixed", dict(scale=1 / 32, ragged=True))]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_refresh_after_commit_equals_rebuild_and_oracle(kap, name, kw):
    import oracle
    from workloads import make_workload
    dev = "cuda"
    w = make_workload(name, device=dev, **kw)
    bt = w.block_table.cpu().numpy()
    L1 = w.ctx_len.cpu().numpy().astype(np.int32)
    rng = np.random.default_rng(11)
    # 17..40 tokens committed per request: the old partial page fills up and at least one new page begins
    L0 = np.array([max(1, int(L) - int(rng.integers(17, 41))) for L in L1], dtype=np.int32)

    def built(ctx):
        s = torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev)
        pool = kap.KVPool(w.K, w.V, w.Hq, s)
        kap.kap_build_summaries(pool, kap.PageMap(w.block_table, torch.as_tensor(ctx, device=dev), w.seq_len0))
        return pool, s

    pool, S = built(L0)
    pages, n_valid = [], []
    for r in range(w.R):
        for j in range(int(L0[r]) // 16, (int(L1[r]) + 15) // 16):
            pages.append(int(bt[r, j]))
            n_valid.append(min(16, int(L1[r]) - 16 * j))
    assert any(n < 16 for n in n_valid) and len(pages) > w.R  # partial pages and page crossings are covered
    kap.kap_refresh_summaries(pool, torch.tensor(pages, dtype=torch.int32, device=dev),
                              torch.tensor(n_valid, dtype=torch.int32, device=dev))
    _, S_full = built(L1)
    torch.cuda.synchronize()
    assert torch.equal(S.view(torch.int32), S_full.view(torch.int32))
    S_orc = oracle.build_summaries(w.K.float().cpu().numpy(), bt, L1)
    S_gpu = S.cpu().numpy()
    for r in range(w.R):
        listed = bt[r, :(int(L1[r]) + 15) // 16]
        assert np.array_equal(S_gpu[listed], S_orc[listed])
    assert kap.kap_device_error() == 0


def test_refresh_reports_bad_entries(kap):
    from workloads import make_workload
    dev = "cuda"
    w = make_workload("tiny", device=dev, ragged=True)
    S = torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev)
    pool = kap.KVPool(w.K, w.V, w.Hq, S)
    page0 = int(w.block_table[0, 0])
    # a page outside the pool, then a count of 0: both skipped and reported; the valid entry is still refreshed
    kap.kap_refresh_summaries(pool, torch.tensor([w.num_pages, page0], dtype=torch.int32, device=dev),
                              torch.tensor([16, 16], dtype=torch.int32, device=dev))
    kap.kap_refresh_summaries(pool, torch.tensor([page0 + 1 if page0 + 1 < w.num_pages else page0 - 1],
                                                 dtype=torch.int32, device=dev),
                              torch.tensor([0], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    err = kap.kap_device_error()
    assert err & 1 and err & 4
    S_full = torch.zeros_like(S)
    kap.kap_build_summaries(kap.KVPool(w.K, w.V, w.Hq, S_full), kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    torch.cuda.synchronize()
    assert torch.equal(S[page0].view(torch.int32), S_full[page0].view(torch.int32))  # page 0 of a prompt is full
    assert kap.kap_device_error() == 0
