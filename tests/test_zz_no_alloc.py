"""The allocation-free proposal entry point (kap_attn_propose_noalloc) against the workspace one and the oracle.

Callers such as a serving host that fixes its device memory budget at start-up, or a plug-in with no access to the
host's allocator, cannot hand the library a freshly allocated workspace; the no-alloc entry point runs the same
kernel on a fixed scratch array inside the library. This file is collected last so that a failure here does not hide
the other tests in a run that stops at the first failure; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw", [("llama", dict(scale=1 / 16)), ("mixed", dict(scale=1 / 32, ragged=True))])
def test_noalloc_matches_workspace_entry_point(kap, name, kw):
    from tests.gpu_helpers import TOL, assert_close_attn, make_cycle, oracle_first_proposal
    from workloads import make_workload
    w = make_workload(name, device="cuda", **kw)
    o_orc, lse_orc = oracle_first_proposal(w)   # before the cycle writes the step token into the pool
    pool, cyc = make_cycle(w)
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    q = w.q_prop[0].clone()
    cyc.plan(w.q_route)
    cyc.append_step(0, q, w.k_new_prop[0], w.v_new_prop[0])
    ref_o = torch.empty_like(cyc.o_prop[0])
    ref_l = torch.empty_like(cyc.lse_prop[0])
    kap.kap_attn_propose(pool, cyc.map_steps[0], cyc.view, q, ref_o, ref_l, cyc.ws_prop)
    torch.cuda.synchronize()
    assert kap.kap_noalloc_scratch_bytes() == 16 << 20
    for call in range(2):   # two calls in a row: the shared scratch must not carry state between calls
        o = torch.full_like(ref_o, float("nan"))
        l = torch.full_like(ref_l, float("nan"))
        kap.kap_attn_propose_noalloc(pool, cyc.map_steps[0], cyc.view, q, o, l)
        torch.cuda.synchronize()
        err = (o.float() - ref_o.float()).abs().max().item()
        lerr = (l - ref_l).abs().max().item()
        assert np.isfinite(err) and err <= TOL[w.dtype], (call, err)
        assert np.isfinite(lerr) and lerr <= 1e-3, (call, lerr)
        # and against the oracle's own first proposal step on the generator's inputs
        assert_close_attn(o.float().cpu().numpy(), o_orc, l.cpu().numpy(), lse_orc, w.dtype, f"noalloc call {call}")
    assert kap.kap_device_error() == 0


def test_noalloc_rejects_shapes_over_the_scratch(kap):
    # 1024 requests x 8 KV heads x 8 query heads per KV head need more partial records than the fixed scratch holds
    need = kap.kap_propose_workspace_size(1024, 8, 64, 128)
    assert need > kap.kap_noalloc_scratch_bytes()
    dev = "cuda"
    K = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device=dev)
    pool = kap.KVPool(K, K.clone(), 64)
    bt = torch.zeros(1024, 1, dtype=torch.int32, device=dev)
    ln = torch.ones(1024, dtype=torch.int32, device=dev)
    pmap = kap.PageMap(bt, ln, ln)
    view = kap.View.empty(1024, 8, 2, dev)
    q = torch.zeros(1024, 64, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(kap.KapError) as e:
        kap.kap_attn_propose_noalloc(pool, pmap, view, q, torch.empty_like(q),
                                     torch.empty(1024, 64, dtype=torch.float32, device=dev))
    assert e.value.status == -3
