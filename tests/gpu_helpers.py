"""Helpers shared by the GPU parity tests: run the library on a workload, and run the oracle on the same inputs.

Only data movement lives here (copies, gathers of one request's pages, slicing); every number the oracle compares
against is computed by the oracle package.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import selected_kv_sparse_gb300 as kap
from workloads import make_workload

PAGE = 16
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}
LSE_TOL = 1e-3


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int32)


def policy_of(w, cap=None):
    a, r, k = (int(x) for x in w.ark[0].tolist())
    same = bool((w.ark == w.ark[0]).all())
    cap = cap if cap is not None else w.sel_cap()
    return kap.AccessPolicy(a, r, k, w.per_kv_head, cap, None if same else w.ark.contiguous())


def make_cycle(w, cap=None, fused=True, overlap=True, ws_pages=0, K=None, V=None):
    """The library's cycle on workload w. ws_pages > 0: the pool tensors K, V carry ws_pages * R extra pages after
    the workload's pool, used as the materialised compact workspace."""
    K = w.K if K is None else K
    V = w.V if V is None else V
    pool = kap.KVPool(K, V, w.Hq, torch.zeros(K.shape[0], w.Hkv, w.d, dtype=torch.float32, device=w.K.device))
    inv = kap.rope_inv_freq(w.d, w.theta, w.K.device)
    pol = policy_of(w, cap)
    cyc = kap.DecodeCycle(pool, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q, inv, policy=pol,
                          spans=w.spans, span_offsets=w.span_offsets, sel_cap=pol.cap, fused=fused, overlap=overlap,
                          workspace_pages=(w.num_pages, ws_pages) if ws_pages else None)
    return pool, cyc


def with_workspace(w, ws_pages):
    """Pool tensors of w followed by R * ws_pages NaN pages (the workspace; NaN shows any read of an unused page)."""
    pad = (w.R * ws_pages,) + tuple(w.K.shape[1:])
    K = torch.cat([w.K, torch.full(pad, float("nan"), dtype=w.K.dtype, device=w.K.device)])
    V = torch.cat([w.V, torch.full(pad, float("nan"), dtype=w.V.dtype, device=w.V.device)])
    return K, V


def oracle_selection(w, S_np, q_route_np):
    """Oracle scores (fixed order) and A/R/K selection, or span selection, as [R][rows][cap] + counts."""
    bt, ctx = i32(w.block_table), i32(w.ctx_len)
    R = w.R
    if w.spans is not None:
        sp = i32(w.spans)
        so = i32(w.span_offsets)
        rows = 1
        sels = []
        for r in range(R):
            N = (int(ctx[r]) + PAGE - 1) // PAGE
            a, rr, _ = (int(x) for x in w.ark[r].tolist())
            sels.append([oracle.select_spans(N, sp[so[r]:so[r + 1]], a, rr)])
    else:
        rows = w.Hkv if w.per_kv_head else 1
        sc, _ = oracle.scores(q_route_np, S_np, bt, ctx, per_head=w.per_kv_head)
        sels = []
        for r in range(R):
            N = (int(ctx[r]) + PAGE - 1) // PAGE
            a, rr, k = (int(x) for x in w.ark[r].tolist())
            sels.append([oracle.topk_ark(sc[r, v], N, a, rr, k) for v in range(rows)])
    cap = max(1, max(len(s) for row in sels for s in row))
    sel = np.zeros((R, rows, cap), np.int32)
    nsel = np.zeros((R, rows), np.int32)
    for r in range(R):
        for v in range(rows):
            sel[r, v, :len(sels[r][v])] = sels[r][v]
            nsel[r, v] = len(sels[r][v])
    return sel, nsel


def run_cycle_and_oracle(w, check_rows=None, nthreads=8, fused=True, ws_pages=0, cap=None):
    """Runs one full cycle on the GPU and the oracle on identical inputs (proposal steps fused with their KV append,
    or as separate append and proposal calls).

    Returns a dict with GPU and oracle results for selection, view, proposal (every step) and verify.
    The oracle sees the pool exactly as the GPU kernels saw it at each point: proposal step i sees the proposal
    tokens 0..i appended (RoPE'd by the oracle itself), verify sees the window tokens appended.
    """
    dev = w.K.device
    Kp, Vp = with_workspace(w, ws_pages) if ws_pages else (w.K, w.V)
    pool, cyc = make_cycle(w, cap=cap, fused=fused, ws_pages=ws_pages, K=Kp, V=Vp)
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    # snapshot inputs before the cycle mutates them (q is rotated in place, the pool receives new tokens)
    K0, V0 = f32(w.K), f32(w.V)
    q_route = w.q_route.clone()
    q_prop_raw, q_ver_raw = f32(w.q_prop), f32(w.q_ver)
    q_prop = w.q_prop.clone()
    q_ver = w.q_ver.clone()
    cyc.run(q_route, q_prop, w.k_new_prop, w.v_new_prop, q_ver, w.k_new_ver, w.v_new_ver)
    torch.cuda.synchronize()
    res = dict(cycle=cyc, pool=pool)
    res["S_gpu"] = pool.k_summary.cpu().numpy()
    bt, ctx, seq0 = i32(w.block_table), i32(w.ctx_len), i32(w.seq_len0)
    S = oracle.build_summaries(K0, bt, ctx)
    res["S_orc"] = S
    sel, nsel = oracle_selection(w, S, f32(w.q_route))
    res["sel_orc"], res["nsel_orc"] = sel, nsel
    if w.spans is None:   # page scores: the score workspace holds them [R][rows][max_pages] after the plan
        rows = w.Hkv if w.per_kv_head else 1
        res["scores_orc"], _ = oracle.scores(f32(w.q_route), S, bt, ctx, per_head=w.per_kv_head)
        mp = int(w.block_table.shape[1])
        res["scores_gpu"] = cyc.ws_score[: w.R * rows * mp * 4].view(torch.float32).view(w.R, rows, mp).cpu().numpy()
    res["sel_gpu"], res["nsel_gpu"] = i32(cyc.sel_ids), i32(cyc.n_sel)
    inv = oracle.inv_freq(w.d, w.theta)
    # proposal steps: oracle appends token i (RoPE'd) at position seq0 + i and attends from there
    K, V = K0.copy(), V0.copy()
    kp, vp = f32(w.k_new_prop), f32(w.v_new_prop)
    res["prop"] = []
    for i in range(w.k_prop):
        pos = seq0 + i
        krot = oracle.rope(kp[i], pos, inv)
        qrot = oracle.rope(q_prop_raw[i], pos, inv)
        for r in range(w.R):
            s = oracle.slot(bt[r], int(pos[r]))
            K[s // PAGE, :, s % PAGE] = krot[r].astype(np.float32) if w.dtype == torch.float32 else \
                torch.from_numpy(krot[r]).to(torch.bfloat16).float().numpy()
            V[s // PAGE, :, s % PAGE] = vp[i, r]
        qin = qrot.astype(np.float32) if w.dtype == torch.float32 else \
            torch.from_numpy(qrot).to(torch.bfloat16).float().numpy()
        out, lse = oracle.attn_propose(qin, K, V, bt, ctx, seq0 + i + 1, sel, nsel, nthreads=nthreads)
        res["prop"].append(dict(o_orc=out, lse_orc=lse, o_gpu=f32(cyc.o_prop[i]), lse_gpu=f32(cyc.lse_prop[i]),
                                q_gpu=None if fused else f32(q_prop[i]), q_orc=qrot))
    # verify: window tokens appended at seq0 .. seq0 + n_q - 1 (overwriting proposal slots)
    qo = i32(w.q_offsets)
    kv_, vv_ = f32(w.k_new_ver), f32(w.v_new_ver)
    posv = np.concatenate([seq0[r] + np.arange(qo[r + 1] - qo[r]) for r in range(w.R)]).astype(np.int32)
    krot = oracle.rope(kv_, posv, inv)
    qrot = oracle.rope(q_ver_raw, posv, inv)
    for r in range(w.R):
        for j in range(qo[r], qo[r + 1]):
            s = oracle.slot(bt[r], int(posv[j]))
            K[s // PAGE, :, s % PAGE] = krot[j].astype(np.float32) if w.dtype == torch.float32 else \
                torch.from_numpy(krot[j]).to(torch.bfloat16).float().numpy()
            V[s // PAGE, :, s % PAGE] = vv_[j]
    qin = qrot.astype(np.float32) if w.dtype == torch.float32 else \
        torch.from_numpy(qrot).to(torch.bfloat16).float().numpy()
    out, lse = oracle.attn_verify(qin, K, V, bt, qo, seq0, nthreads=nthreads)
    res["ver"] = dict(o_orc=out, lse_orc=lse, o_gpu=f32(cyc.o_ver), lse_gpu=f32(cyc.lse_ver))
    res["K_after_orc"], res["K_after_gpu"] = K, f32(Kp[:w.num_pages])
    res["V_after_orc"], res["V_after_gpu"] = V, f32(Vp[:w.num_pages])
    res["K_pool"], res["V_pool"] = Kp, Vp
    return res


def run_cycle_per_request(w, nthreads=16, fused=True):
    """One full cycle on the GPU, then the oracle request by request on that request's own pages only, for pools
    too large to copy to the host (the mixed batch's 2^20-page pool holds 64 GiB).

    Each request's pages (its block-table row, prompt and tail) are copied to the host before the cycle, in the pool
    dtype; the oracle then runs on them with a local table 0..n-1, appending the cycle's tokens itself. Yields, per
    request r, a dict of GPU and oracle results: summaries, scores, selection, view row, slots, appended K/V, every
    proposal step and the verify rows.
    """
    pool, cyc = make_cycle(w, fused=fused)
    kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
    bt, ctx, seq0 = i32(w.block_table), i32(w.ctx_len), i32(w.seq_len0)
    qo = i32(w.q_offsets)
    horizon = max(w.k_prop, int(w.n_q.max()))
    npg = [(int(ctx[r]) + horizon + PAGE - 1) // PAGE for r in range(w.R)]
    snap = []
    for r in range(w.R):   # the generator's pages of request r, before the cycle writes into them
        idx = w.block_table[r, :npg[r]].to(torch.int64)
        snap.append((w.K.index_select(0, idx).cpu(), w.V.index_select(0, idx).cpu()))
    q_route_np = f32(w.q_route)
    q_prop_raw, q_ver_raw = f32(w.q_prop), f32(w.q_ver)
    kp, vp = f32(w.k_new_prop), f32(w.v_new_prop)
    kv_, vv_ = f32(w.k_new_ver), f32(w.v_new_ver)
    cyc.run(w.q_route.clone(), w.q_prop.clone(), w.k_new_prop, w.v_new_prop, w.q_ver.clone(), w.k_new_ver,
            w.v_new_ver)
    torch.cuda.synchronize()
    mp = int(w.block_table.shape[1])
    rows = cyc.rows
    scores_gpu = cyc.ws_score[: w.R * rows * mp * 4].view(torch.float32).view(w.R, rows, mp).cpu().numpy()
    sel_gpu, nsel_gpu = i32(cyc.sel_ids), i32(cyc.n_sel)
    vbt, vlp = i32(cyc.view.block_table), i32(cyc.view.logical_page)
    vn, vns = i32(cyc.view.n_entries), i32(cyc.view.n_selected)
    slots = cyc.slots_prop.cpu().numpy().reshape(w.R, cyc.horizon)
    o_prop, lse_prop = f32(cyc.o_prop), f32(cyc.lse_prop)
    o_ver, lse_ver = f32(cyc.o_ver), f32(cyc.lse_ver)
    inv = oracle.inv_freq(w.d, w.theta)
    rnd = (lambda x: x.astype(np.float32)) if w.dtype == torch.float32 else \
        (lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).float().numpy())
    for r in range(w.R):
        N = (int(ctx[r]) + PAGE - 1) // PAGE
        idx = w.block_table[r, :npg[r]].to(torch.int64)
        K = snap[r][0].float().numpy()
        V = snap[r][1].float().numpy()
        lbt = np.arange(npg[r], dtype=np.int32)[None]
        lctx, lseq = ctx[r:r + 1], seq0[r:r + 1]
        out = dict(r=r, N=N)
        out["S_gpu"] = pool.k_summary.index_select(0, idx[:N]).cpu().numpy()
        S = oracle.build_summaries(K, lbt, lctx)
        out["S_orc"] = S[:N]
        if w.spans is None:
            sc, _ = oracle.scores(q_route_np[r:r + 1], S, lbt, lctx, per_head=w.per_kv_head)
            out["scores_orc"], out["scores_gpu"] = sc[0, :, :N], scores_gpu[r, :, :N]
            a, rr, k = (int(x) for x in w.ark[r].tolist())
            sels = [oracle.topk_ark(sc[0, v], N, a, rr, k) for v in range(rows)]
        else:
            so = i32(w.span_offsets)
            a, rr, _ = (int(x) for x in w.ark[r].tolist())
            sels = [oracle.select_spans(N, i32(w.spans)[so[r]:so[r + 1]], a, rr)]
        cap = max(1, max(len(x) for x in sels))
        sel = np.zeros((1, rows, cap), np.int32)
        nsel = np.zeros((1, rows), np.int32)
        for v, x in enumerate(sels):
            sel[0, v, :len(x)] = x
            nsel[0, v] = len(x)
        out["sel_orc"], out["nsel_orc"] = sel[0], nsel[0]
        out["sel_gpu"], out["nsel_gpu"] = sel_gpu[r], nsel_gpu[r]
        out["view"] = []
        for v in range(rows):
            cbt, clog, ns = oracle.compile_view_row(bt[r], int(ctx[r]), int(seq0[r]), cyc.horizon,
                                                    sels[v])
            out["view"].append(((cbt, clog, ns), (vbt[r, v, :vn[r, v]], vlp[r, v, :vn[r, v]], vns[r, v])))
        out["slots"] = [(slots[r, i], oracle.slot(bt[r], int(seq0[r]) + i)) for i in range(cyc.horizon)]
        # proposal steps: the oracle appends step token i at seq0 + i (local slot) and attends from there
        out["prop"] = []
        for i in range(w.k_prop):
            pos = np.array([seq0[r] + i], np.int32)
            krot = oracle.rope(kp[i, r:r + 1], pos, inv)
            qrot = oracle.rope(q_prop_raw[i, r:r + 1], pos, inv)
            s = oracle.slot(lbt[0], int(pos[0]))
            K[s // PAGE, :, s % PAGE] = rnd(krot[0])
            V[s // PAGE, :, s % PAGE] = vp[i, r]
            o, l = oracle.attn_propose(rnd(qrot), K, V, lbt, lctx, lseq + i + 1, sel, nsel, nthreads=nthreads)
            out["prop"].append((o_prop[i, r], o[0], lse_prop[i, r], l[0]))
        # verify window at seq0 .. seq0 + n_q - 1
        nq = int(qo[r + 1] - qo[r])
        posv = (seq0[r] + np.arange(nq)).astype(np.int32)
        krot = oracle.rope(kv_[qo[r]:qo[r + 1]], posv, inv)
        qrot = oracle.rope(q_ver_raw[qo[r]:qo[r + 1]], posv, inv)
        for j in range(nq):
            s = oracle.slot(lbt[0], int(posv[j]))
            K[s // PAGE, :, s % PAGE] = rnd(krot[j])
            V[s // PAGE, :, s % PAGE] = vv_[qo[r] + j]
        o, l = oracle.attn_verify(rnd(qrot), K, V, lbt, np.array([0, nq], np.int32), lseq, nthreads=nthreads)
        out["ver"] = (o_ver[qo[r]:qo[r + 1]], o, lse_ver[qo[r]:qo[r + 1]], l)
        out["K_after"] = (w.K.index_select(0, idx).float().cpu().numpy(), K)
        out["V_after"] = (w.V.index_select(0, idx).float().cpu().numpy(), V)
        out["k_in_max"] = max(float(np.abs(kp[:, r]).max()), float(np.abs(kv_[qo[r]:qo[r + 1]]).max()))
        yield out


def oracle_first_proposal(w, nthreads=8):
    """The oracle's first proposal step on workload w, from the generator's tensors alone: summaries, selection,
    the step token's K (RoPE at seq_len0) and V written into a copy of the pool, the query rotated at the same
    position, then attention over the selection. Returns (o, lse); the inputs must not yet be modified by a cycle."""
    K, V = f32(w.K), f32(w.V)
    bt, ctx, seq0 = i32(w.block_table), i32(w.ctx_len), i32(w.seq_len0)
    S = oracle.build_summaries(K, bt, ctx)
    sel, nsel = oracle_selection(w, S, f32(w.q_route))
    inv = oracle.inv_freq(w.d, w.theta)
    krot = oracle.rope(f32(w.k_new_prop[0]), seq0, inv)
    qrot = oracle.rope(f32(w.q_prop[0]), seq0, inv)
    vp = f32(w.v_new_prop[0])
    rnd = (lambda x: x.astype(np.float32)) if w.dtype == torch.float32 else \
        (lambda x: torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    for r in range(w.R):
        s = oracle.slot(bt[r], int(seq0[r]))
        K[s // PAGE, :, s % PAGE] = rnd(krot[r])
        V[s // PAGE, :, s % PAGE] = vp[r]
    return oracle.attn_propose(rnd(qrot), K, V, bt, ctx, seq0 + 1, sel, nsel, nthreads=nthreads)


def assert_close_attn(o_gpu, o_orc, lse_gpu, lse_orc, dtype, what=""):
    tol = TOL[dtype]
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    err = np.abs(o_gpu.astype(np.float64) - o_orc).max()
    assert err <= tol, f"{what}: max |o - oracle| = {err:.3e} > {tol}"
    lerr = np.abs(lse_gpu.astype(np.float64) - lse_orc).max()
    assert lerr <= LSE_TOL, f"{what}: max |lse - oracle| = {lerr:.3e} > {LSE_TOL}"
