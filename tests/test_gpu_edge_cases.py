"""Degenerate shapes and device-side error detection, through the C ABI against the oracle.

Prompts of 1, 16, 17 and 40 tokens (a row of one page, N <= a + r), recency-only selection (k = 0), a k larger than
the middle of the row (every page kept), and a page id outside the pool in a view and in a block table: the kernels
must skip that access, record device error bit 1, and leave the context usable for the next call.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _short(ark):
    from workloads import make_workload
    w = make_workload("llama", device="cuda", scale=1 / 64, poison=True)   # 4 requests, pages for 512 tokens each
    lens = torch.tensor([1, 16, 17, 40], dtype=torch.int32, device="cuda")
    w.ctx_len = lens.clone()
    w.seq_len0 = lens.clone()
    w.ark = torch.tensor([ark] * w.R, dtype=torch.int32, device="cuda")
    w.needles = [[] for _ in range(w.R)]
    return w


@pytest.mark.parametrize("ark", [(1, 2, 5), (1, 2, 0), (1, 2, 10000), (0, 0, 1)],
                         ids=["A1R2K5", "A1R2K0", "A1R2K10000", "A0R0K1"])
def test_short_prompts_and_degenerate_splits(kap, ark):
    from tests.gpu_helpers import assert_close_attn, run_cycle_and_oracle
    w = _short(ark)
    # the row capacity the API asks for: a + r + k, or the whole table when that is smaller
    cap = min(sum(ark), int(w.block_table.shape[1]))
    res = run_cycle_and_oracle(w, cap=cap)
    assert np.array_equal(res["nsel_gpu"], res["nsel_orc"])
    for r in range(w.R):
        for v in range(res["nsel_orc"].shape[1]):
            n = int(res["nsel_orc"][r, v])
            assert np.array_equal(res["sel_gpu"][r, v, :n], res["sel_orc"][r, v, :n])
    for st in res["prop"]:
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, "propose")
    v = res["ver"]
    assert_close_attn(v["o_gpu"], v["o_orc"], v["lse_gpu"], v["lse_orc"], w.dtype, "verify")
    assert kap.kap_device_error() == 0


def test_short_prompts_in_a_large_batch(kap):
    """More than 8 requests: the score kernel's CTAs scan the requests' chunk counts and take contiguous item ranges
    that cross requests. Prompts of 1, 16, 17 and 40 tokens among ragged ones of up to 2K; scores, selections,
    views and attention against the oracle."""
    from tests.gpu_helpers import assert_close_attn, run_cycle_and_oracle
    from workloads import make_workload
    w = make_workload("mixed", device="cuda", scale=1 / 64, batch=12, ragged=True, poison=True)
    lens = w.ctx_len.clone()
    for r, n in ((0, 1), (3, 16), (5, 17), (7, 40)):
        lens[r] = n
    w.ctx_len = lens.clone()
    w.seq_len0 = lens.clone()
    w.needles = [[] for _ in range(w.R)]
    res = run_cycle_and_oracle(w)
    ctx = w.ctx_len.cpu().numpy()
    for r in range(w.R):   # every prompt page's score, bit for bit
        N = (int(ctx[r]) + 15) // 16
        g, o = res["scores_gpu"][r, :, :N], res["scores_orc"][r, :, :N]
        assert np.array_equal(g.view(np.uint32), o.view(np.uint32)), r
    assert np.array_equal(res["nsel_gpu"], res["nsel_orc"])
    for r in range(w.R):
        for v in range(res["nsel_orc"].shape[1]):
            n = int(res["nsel_orc"][r, v])
            assert np.array_equal(res["sel_gpu"][r, v, :n], res["sel_orc"][r, v, :n])
    for st in res["prop"]:
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, "propose")
    v = res["ver"]
    assert_close_attn(v["o_gpu"], v["o_orc"], v["lse_gpu"], v["lse_orc"], w.dtype, "verify")
    assert kap.kap_device_error() == 0


def test_bad_page_ids_are_skipped_and_reported(kap):
    from tests.gpu_helpers import make_cycle
    from workloads import make_workload
    w = make_workload("llama", device="cuda", scale=1 / 32, poison=False)
    pool, cyc = make_cycle(w)
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    cyc.plan(w.q_route)
    torch.cuda.synchronize()
    assert kap.kap_device_error() == 0
    # a view entry (the anchor page of request 0, KV head 0) outside the pool
    saved = cyc.view.block_table[0, 0, 0].item()
    cyc.view.block_table[0, 0, 0] = w.num_pages + 5
    cyc.propose_step(0, w.q_prop[0].clone(), w.k_new_prop[0], w.v_new_prop[0])
    torch.cuda.synchronize()
    assert kap.kap_device_error() & 1
    cyc.view.block_table[0, 0, 0] = saved
    # the context still works: the same step again, clean
    cyc.propose_step(0, w.q_prop[0].clone(), w.k_new_prop[0], w.v_new_prop[0])
    torch.cuda.synchronize()
    assert kap.kap_device_error() == 0
    # a full block-table entry (page 3 of request 1) outside the pool, read by verification
    cyc.append_window(w.q_ver.clone(), w.k_new_ver, w.v_new_ver)
    saved = w.block_table[1, 3].item()
    w.block_table[1, 3] = -2
    cyc.verify(w.q_ver.clone())
    torch.cuda.synchronize()
    assert kap.kap_device_error() & 1
    w.block_table[1, 3] = saved
    cyc.verify(w.q_ver.clone())
    torch.cuda.synchronize()
    assert kap.kap_device_error() == 0
