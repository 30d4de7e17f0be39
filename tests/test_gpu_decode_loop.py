"""EarlySelectKV decode loop over 1024 generated tokens (batch 1 and 8, prompts of 2555 tokens): every step re-routes
on its own proxy query, appends one token at the committed length and attends over the selected pages plus every
generated token, so the view's tail grows by a page every 16 steps. The oracle replays the loop on the generator's
inputs, appending each token itself; it is compared with the library at every step that opens or closes a page and
at a seeded sample of the others (selection, view and attention), and over the whole pool after the last step."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

STEPS = 1024


@pytest.mark.parametrize("batch", [1, 8])
def test_decode_loop_1024_steps(kap, batch):
    import oracle
    from tests.gpu_helpers import PAGE, assert_close_attn, f32, i32, policy_of
    from workloads import make_workload
    w = make_workload("early", device="cuda", scale=1 / 16, batch=batch, ragged=True, k_prop_override=STEPS)
    R, rows = w.R, w.Hkv
    bt, ctx, seq0 = i32(w.block_table), i32(w.ctx_len), i32(w.seq_len0)
    K, V = f32(w.K), f32(w.V)               # the oracle's copy, before the loop writes into the pool
    q_route, q_prop = f32(w.q_route_steps), f32(w.q_prop)
    kp, vp = f32(w.k_new_prop), f32(w.v_new_prop)

    pool = kap.KVPool(w.K, w.V, w.Hq, torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device="cuda"))
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    pol = policy_of(w)
    loop = kap.DecodeLoop(pool, w.block_table, w.ctx_len, w.seq_len0, STEPS, kap.rope_inv_freq(w.d, w.theta, "cuda"),
                          pol)
    hist_sel = torch.zeros((STEPS,) + tuple(loop.sel_ids.shape), dtype=torch.int32, device="cuda")
    hist_nsel = torch.zeros((STEPS,) + tuple(loop.n_sel.shape), dtype=torch.int32, device="cuda")
    hist_vbt = torch.zeros((STEPS,) + tuple(loop.view.block_table.shape), dtype=torch.int32, device="cuda")
    hist_vlp = torch.zeros_like(hist_vbt)
    hist_vn = torch.zeros((STEPS,) + tuple(loop.view.n_entries.shape), dtype=torch.int32, device="cuda")
    for t in range(STEPS):
        loop.plan(w.q_route_steps[t])
        hist_sel[t].copy_(loop.sel_ids)
        hist_nsel[t].copy_(loop.n_sel)
        hist_vbt[t].copy_(loop.view.block_table)
        hist_vlp[t].copy_(loop.view.logical_page)
        hist_vn[t].copy_(loop.view.n_entries)
        loop.propose_step(0, w.q_prop[t], w.k_new_prop[t], w.v_new_prop[t])
        loop.advance()
    torch.cuda.synchronize()
    assert kap.kap_device_error() == 0
    o_gpu, lse_gpu = f32(loop.o), f32(loop.lse)
    sel_g, nsel_g = i32(hist_sel), i32(hist_nsel)
    vbt_g, vlp_g, vn_g = i32(hist_vbt), i32(hist_vlp), i32(hist_vn)

    rng = np.random.default_rng(0x4B4150 + batch)
    check = {0, STEPS - 1}
    for t in range(STEPS):
        if any((int(seq0[r]) + t) % PAGE in (0, PAGE - 1) for r in range(R)):
            check.add(t)
    check |= set(int(x) for x in rng.choice(STEPS, 24, replace=False))
    crossings = sum(1 for t in range(STEPS) if (int(seq0[0]) + t) % PAGE == 0)
    assert crossings == STEPS // PAGE

    inv = oracle.inv_freq(w.d, w.theta)
    S = oracle.build_summaries(K, bt, ctx)   # prompt pages only: generated tokens never enter a summary
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).float().numpy()  # noqa: E731
    for t in range(STEPS):
        pos = (seq0 + t).astype(np.int32)
        krot = oracle.rope(kp[t], pos, inv)
        for r in range(R):
            s = oracle.slot(bt[r], int(pos[r]))
            K[s // PAGE, :, s % PAGE] = bf(krot[r])
            V[s // PAGE, :, s % PAGE] = vp[t, r]
        if t not in check:
            continue
        sc, _ = oracle.scores(q_route[t], S, bt, ctx, per_head=True)
        cap = loop.sel_cap
        sel = np.zeros((R, rows, cap), np.int32)
        nsel = np.zeros((R, rows), np.int32)
        for r in range(R):
            N = (int(ctx[r]) + PAGE - 1) // PAGE
            a, rr, k = (int(x) for x in w.ark[r].tolist())
            for v in range(rows):
                x = oracle.topk_ark(sc[r, v], N, a, rr, k)
                sel[r, v, :len(x)] = x
                nsel[r, v] = len(x)
                assert nsel_g[t, r, v] == len(x) and np.array_equal(sel_g[t, r, v, :len(x)], x), (t, r, v)
                cbt, clog, _ = oracle.compile_view_row(bt[r], int(ctx[r]), int(pos[r]), 1, x)
                assert vn_g[t, r, v] == len(cbt), (t, r, v)
                assert np.array_equal(vbt_g[t, r, v, :len(cbt)], cbt) and np.array_equal(vlp_g[t, r, v, :len(clog)],
                                                                                          clog), (t, r, v)
        qrot = bf(oracle.rope(q_prop[t], pos, inv))
        o, lse = oracle.attn_propose(qrot, K, V, bt, ctx, seq0 + t + 1, sel, nsel, nthreads=8)
        assert_close_attn(o_gpu[t], o, lse_gpu[t], lse, w.dtype, f"decode step {t}")
    # the whole pool after the loop: every generated token's K (RoPE at its position) and V in its slot
    Kg, Vg = f32(w.K), f32(w.V)
    assert np.array_equal(np.isnan(Kg), np.isnan(K)) and np.array_equal(np.isnan(Vg), np.isnan(V))
    m = ~np.isnan(K)
    ulp = np.maximum(np.abs(K[m]), 1e-30) * 2.0 ** -7
    assert (np.abs(Kg[m] - K[m]) <= 2 * ulp + 2.0 ** -19 * float(np.abs(kp).max())).all()
    assert np.array_equal(Vg[~np.isnan(V)], V[~np.isnan(V)])


def test_decode_loop_side_flow_in_graphs_equals_eager(kap):
    """The loop over a stack of layers with each next layer's routing on a second stream, captured as CUDA graphs of
    16 steps and replayed, must give bit for bit the outputs of the same steps run eagerly one layer after another.
    The view changes at every step here (a new proxy query, a growing tail), so a proposal that read its view before
    the routing that writes it had finished would show."""
    from tests.gpu_helpers import policy_of
    from workloads import make_workload
    steps, layers_n, chunk = 64, 3, 16

    def build():
        loops, ins = [], []
        for l in range(layers_n):
            w = make_workload("early", device="cuda", scale=1 / 16, batch=2, ragged=True, seed_offset=l,
                              k_prop_override=steps)
            pool = kap.KVPool(w.K, w.V, w.Hq,
                              torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device="cuda"))
            kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
            loops.append(kap.DecodeLoop(pool, w.block_table, w.ctx_len, w.seq_len0, steps,
                                        kap.rope_inv_freq(w.d, w.theta, "cuda"), policy_of(w)))
            ins.append(w)
        return loops, ins

    ref, ref_in = build()
    for t in range(steps):
        for lp, w in zip(ref, ref_in):
            lp.plan(w.q_route_steps[t])
            lp.propose_step(0, w.q_prop[t], w.k_new_prop[t], w.v_new_prop[t])
            lp.advance()
    torch.cuda.synchronize()
    loops, ins = build()
    flow = kap.SideFlowDecode(loops)

    def run(t0, t1):
        for t in range(t0, t1):
            flow.step([w.q_route_steps[t] for w in ins], [w.q_prop[t] for w in ins],
                      [w.k_new_prop[t] for w in ins], [w.v_new_prop[t] for w in ins])
            for lp in loops:
                lp.advance()
    run(0, chunk)   # eager once (kernel attributes, stream set-up), then capture every chunk and replay the loop
    torch.cuda.synchronize()
    for lp in loops:
        lp.reset()
    graphs = []
    for c0 in range(0, steps, chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(c0, c0 + chunk)
        graphs.append(g)
    for lp in loops:
        lp.o.zero_()
        lp.lse.zero_()
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    for l, (a, b) in enumerate(zip(loops, ref)):
        assert torch.equal(a.o.view(torch.int16), b.o.view(torch.int16)), l
        assert torch.equal(a.lse.view(torch.int32), b.lse.view(torch.int32)), l
    assert kap.kap_device_error() == 0
