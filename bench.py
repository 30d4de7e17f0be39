#!/usr/bin/env python
"""Benchmark of the selected-KV sparse decode hot path on GB300.

One step = one proposal/verification cycle of the whole hot path over `--layers` independent attention layers
(replicas with their own KV pools), on the Llama-3-8B-shaped workload: 4 requests x 32768-token prompts, Hq=32,
Hkv=8, d=128, bf16 KV, per-KV-head K-summary scoring with A1R2K125 selection (s = 6.25%), 4 proposal steps (q=1)
and a verify window of 4 (causal). Per layer and cycle: scoring, then top-K with the view compilation (and the slot
mapping of the cycle's new tokens) in the same kernel, then 4 proposal steps, each one kernel that appends the step
token's KV and attends over the view, then window append + verification. --unfused runs the separate calls: score,
top-K, view; a KV-append kernel and a proposal kernel per step.

Output: one JSON line (rank 0). `value` is the algorithmic HBM bytes of every hot-path kernel in a step divided by
the device time of the step (GB/s, whole job); the phase times come from CUDA events recorded between CUDA-graph
replays of each phase on the launch stream. `--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse paged attention HBM GB/s (% of roofline); proposal & verify steps/s"
PAGE = 16
CONFIG = "llama"
WORKLOAD = ("Llama-3-8B-shaped attention layer: 4 requests x 32768-token prompts (2048 pages of 16), Hq=32, Hkv=8, "
            "d=128, bf16 KV, fp32 accumulation, per-KV-head A1R2K125 (s=6.25%), 16 needle pages/request, "
            "4 proposal steps (q=1) + verify window 4 (causal)")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["kap", "reference"], default="kap")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prior", action="store_true", help="skip the external-prior selection timing")
    ap.add_argument("--no-accept", action="store_true", help="skip the acceptance and commit timing")
    ap.add_argument("--no-materialize", action="store_true", help="skip the materialised-workspace timing")
    ap.add_argument("--no-side-flow", action="store_true", help="skip the EarlySelectKV side-flow timing")
    ap.add_argument("--no-decode-loop", action="store_true", help="skip the 1024-step EarlySelectKV decode loop")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the long-context and mixed-batch workload lines")
    ap.add_argument("--unfused", action="store_true", help="separate KV-append and proposal launches per step")
    ap.add_argument("--no-overlap", action="store_true",
                    help="proposal kernels wait for the previous kernel before reading their view")
    ap.add_argument("--clock-log", default=None, help="CSV file for the nvidia-smi samples of the timed region")
    return ap.parse_args(argv)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def reduce_max(value: float, dist=None) -> float:
    """Max of a per-rank scalar over all ranks (timing only, not on the data path)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, dist=None) -> float:
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------- clock sampling
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path=None):
        import tempfile
        self.index = index
        self.proc = None
        if path is None:
            fd, path = tempfile.mkstemp(prefix=f"kap_clocks{index}_", suffix=".csv")
            os.close(fd)
        self.path = path

    def start(self):
        if os.path.dirname(self.path):
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


# --------------------------------------------------------------------------------------------- byte model
def step_bytes(w, cyc, sel_ids, n_sel):
    """Algorithmic HBM bytes of one cycle on one layer, per kernel family:
    scores read every prompt page's fp32 summary; proposal step i reads K and V of every visible token of the
    view (selected prompt tokens + generated tokens up to the step's position); verification reads K and V of
    every position up to the last window row; appends write K and V of the new tokens."""
    import numpy as np
    kv_tok = w.d * 2 * 2  # bytes of K+V of one token of one KV head (bf16)
    ctx = w.ctx_len.cpu().numpy().astype(np.int64)
    seq0 = w.seq_len0.cpu().numpy().astype(np.int64)
    N = (ctx + PAGE - 1) // PAGE
    score = int((N * w.Hkv * w.d * 4).sum())
    sel = sel_ids.cpu().numpy()
    ns = n_sel.cpu().numpy()
    rows = sel.shape[1]
    prop = []
    for i in range(w.k_prop):
        tot = 0
        for r in range(w.R):
            for h in range(w.Hkv):
                v = 0 if rows == 1 else h
                pages = sel[r, v, :ns[r, v]]
                tok = np.minimum(PAGE, ctx[r] - PAGE * pages.astype(np.int64)).clip(min=0).sum()
                tok += (seq0[r] + i + 1) - ctx[r]   # generated positions ctx .. seq0 + i
                tot += int(tok) * kv_tok
        prop.append(tot)
    nq = w.n_q.cpu().numpy().astype(np.int64)
    ver = int(((seq0 + nq) * w.Hkv * kv_tok).sum())
    app = int((w.k_prop * w.R + nq.sum()) * w.Hkv * w.d * 2 * 2)
    return dict(score=score, propose=prop, verify=ver, append=app)


# ----------------------------------------------------------------------------------- external-prior selection
PRIOR_LAYERS = 32   # layers of a baked prior (block_affinities[L][H][N]); H is the KV head count


def time_prior(layers, steps: int, hbm_peak: float, dev):
    """Times kap_prior_topk (KRI page, prior schema: pool a baked block_affinities[L][H][N] over layers and heads,
    then take each request's A/R/K top-K) on every layer's page map, three distinct priors per layer so that the
    priors read per replay exceed L2. Returns per-call time, the prior bytes a call reads and its GB/s."""
    import torch
    import selected_kv_sparse_gb300 as kap
    from workloads import make_prior
    calls = []
    for li, (w, _, _) in enumerate(layers):
        a, r, k = (int(x) for x in w.ark[0].tolist())
        cap = int(w.sel_cap())
        pol = kap.AccessPolicy(a, r, k, False, cap)
        pmap = kap.PageMap(w.block_table, w.ctx_len)
        max_pages = int(w.block_table.shape[1])
        for rep in range(3):
            aff = make_prior(w, PRIOR_LAYERS, device=dev, seed_offset=li * 3 + rep)
            sel = torch.zeros((w.R, 1, cap), dtype=torch.int32, device=dev)
            nsel = torch.zeros((w.R, 1), dtype=torch.int32, device=dev)
            ws = torch.zeros(kap.kap_score_workspace_size(w.R, 1, max_pages) // 4, dtype=torch.float32, device=dev)
            calls.append((pmap, aff, pol, sel, nsel, ws))

    def run():
        for pmap, aff, pol, sel, nsel, ws in calls:
            kap.kap_prior_topk(pmap, aff, pol, sel, nsel, ws)
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    n = max(3, min(steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (n * len(calls))
    # algorithmic bytes: every prompt page's L*H affinities of every request
    import numpy as np
    w0 = layers[0][0]
    N = ((w0.ctx_len.cpu().numpy().astype(np.int64) + PAGE - 1) // PAGE)
    b = int(N.sum()) * PRIOR_LAYERS * w0.Hkv * 4
    total = sum(c[1].numel() * 4 for c in calls)
    return {"us_per_call": us, "bytes_per_call": b, "gbs": b / (us * 1e-6) / 1e9,
            "pct_of_roofline": 100 * b / (us * 1e-6) / 1e9 / hbm_peak, "prior_layers": PRIOR_LAYERS,
            "l2": f"{len(calls)} distinct priors, {total / 1e6:.0f} MB per replay"}


# ------------------------------------------------------------------------------ EarlySelectKV side flow
def time_side_flow(steps: int, dev, hbm_peak: float, layers_n: int = 8):
    """EarlySelectKV-shaped decode steps (40960-token prompts, Hq 32, Hkv 8, d 128, A0R0K8 per KV head on a proxy
    query = q + N(0, 0.3^2)) over a stack of layers, batch 1 and 8: routing (scores, top-K, view) and the step's
    append + proposal attention per layer, run in turn on one stream or with the next layer's routing on a second
    stream (SideFlowDecode). Each schedule is one CUDA graph per decode step."""
    import torch
    import selected_kv_sparse_gb300 as kap
    from workloads import make_workload
    out = {}
    for batch in (1, 8):
        layers = []
        for l in range(layers_n):
            w = make_workload("early", device=dev, batch=batch, seed_offset=100 + l, poison=False)
            pool = kap.KVPool(w.K, w.V, w.Hq, torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev))
            kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
            a, r, k = (int(x) for x in w.ark[0].tolist())
            cyc = kap.DecodeCycle(pool, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q,
                                  kap.rope_inv_freq(w.d, w.theta, dev), policy=kap.AccessPolicy(a, r, k, True, w.sel_cap()))
            layers.append((w, cyc))
        flow = kap.SideFlowDecode([c for _, c in layers])
        args = ([w.q_route for w, _ in layers], [w.q_prop[0] for w, _ in layers],
                [w.k_new_prop[0] for w, _ in layers], [w.v_new_prop[0] for w, _ in layers])
        res = {}
        for name, ov in (("sequential", False), ("side_flow", True)):
            flow.step(*args, overlap=ov)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                flow.step(*args, overlap=ov)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            n = max(3, min(steps, 50))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            res[name] = e0.elapsed_time(e1) * 1e3 / n
        # algorithmic bytes of one decode step over all layers: the summaries the routing scores (one fp32 summary
        # per prompt page and KV head), the K and V of every token the proposal attends to, the step token written
        by = [step_bytes(w, c, c.sel_ids, c.n_sel) for w, c in layers]
        b_step = sum(b["score"] + b["propose"][0] + w.R * w.Hkv * w.d * 2 * 2 for b, (w, _) in zip(by, layers))
        b_att = sum(b["propose"][0] for b in by)
        t = res["side_flow"] * 1e-6
        out[f"batch{batch}"] = {"us_per_step_sequential": res["sequential"], "us_per_step_side_flow": res["side_flow"],
                                "decode_steps_per_s": 1e6 / res["side_flow"],
                                "speedup": res["sequential"] / res["side_flow"],
                                "bytes_per_step": b_step, "attention_bytes_per_step": b_att,
                                "gbs": b_step / t / 1e9, "pct_of_roofline": 100 * b_step / t / 1e9 / hbm_peak}
        del layers, flow
        torch.cuda.empty_cache()
    out["layers"] = layers_n
    out["workload"] = ("EarlySelectKV-shaped: 40960-token prompts, Hq 32, Hkv 8, d 128, A0R0K8 per KV head on a "
                       "proxy query; a step = routing + append + proposal attention per layer")
    return out


# ------------------------------------------------------------------------ EarlySelectKV 1024-step decode loop
def time_decode_loop(dev, hbm_peak: float, steps: int = 1024, layers_n: int = 8, chunk: int = 128, reps: int = 2):
    """EarlySelectKV decode over `steps` generated tokens (40960-token prompts, Hq 32, Hkv 8, d 128, A0R0K8 per KV
    head on each step's own noisy proxy query), batch 1 and 8, over a stack of `layers_n` layers: every step routes
    and then appends its token and attends, layer after layer, with the next layer's routing on a second stream
    (SideFlowDecode over DecodeLoop). The loop is captured as CUDA graphs of `chunk` steps and timed whole.
    Algorithmic bytes of step t per layer and request: the summaries the routing scores (N * Hkv * d * 4), the K
    and V of the 8 selected pages and of the t + 1 generated tokens, and the step token written."""
    import torch
    import selected_kv_sparse_gb300 as kap
    from workloads import make_workload
    out = {}
    for batch in (1, 8):
        loops, ins = [], []
        for l in range(layers_n):
            w = make_workload("early", device=dev, batch=batch, seed_offset=400 + l, poison=False,
                              k_prop_override=steps)
            pool = kap.KVPool(w.K, w.V, w.Hq, torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev))
            kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
            loops.append(kap.DecodeLoop(pool, w.block_table, w.ctx_len, w.seq_len0, steps,
                                        kap.rope_inv_freq(w.d, w.theta, dev), policy_of(w)))
            ins.append(w)
        flow = kap.SideFlowDecode(loops)

        def run(t0, t1):
            for t in range(t0, t1):
                flow.step([w.q_route_steps[t] for w in ins], [w.q_prop[t] for w in ins],
                          [w.k_new_prop[t] for w in ins], [w.v_new_prop[t] for w in ins])
                for lp in loops:
                    lp.advance()
        for lp in loops:
            lp.reset()
        run(0, steps)   # eager pass
        torch.cuda.synchronize()
        graphs = []
        for lp in loops:
            lp.reset()
        for c0 in range(0, steps, chunk):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run(c0, min(steps, c0 + chunk))
            graphs.append(g)
        for g in graphs:   # warm-up: one whole loop
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for g in graphs:
                g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
        w = ins[0]
        N = (int(w.ctx_len[0]) + PAGE - 1) // PAGE
        kv_tok = w.d * 2 * 2
        sel_tok = 8 * PAGE
        per_req = sum(N * w.Hkv * w.d * 4 + (sel_tok + t + 1) * w.Hkv * kv_tok + w.Hkv * kv_tok for t in range(steps))
        b = per_req * w.R * layers_n / steps     # average bytes of one decode step (all layers)
        out[f"batch{batch}"] = {"us_per_step": us, "decode_steps_per_s": 1e6 / us, "tokens_per_s": 1e6 / us * w.R,
                                "bytes_per_step": b, "gbs": b / (us * 1e-6) / 1e9,
                                "pct_of_roofline": 100 * b / (us * 1e-6) / 1e9 / hbm_peak}
        del loops, ins, flow, graphs
        torch.cuda.empty_cache()
    out.update(layers=layers_n, steps=steps, graph_chunk=chunk, reps=reps,
               workload="EarlySelectKV-shaped decode: 40960-token prompts, Hq 32, Hkv 8, d 128, A0R0K8 per KV head "
                        "re-routed every step on that step's proxy query (q + N(0, 0.3^2)), 1024 generated tokens "
                        "appended one per step; a step = routing + append + attention on every layer, the next "
                        "layer's routing on a second stream")
    return out


# --------------------------------------------------------------------------- materialised compact workspace
def time_materialize(layers, steps: int, hbm_peak: float, dev):
    """Times kap_materialize_view (KAP paper, compiler: the selected pages copied into a compact workspace) on every
    layer's compiled view, and the first proposal step over the materialised views, each as a CUDA graph over the
    layers. Every layer gets a copy of its pool followed by R * cap workspace pages."""
    import torch
    import selected_kv_sparse_gb300 as kap
    import numpy as np
    mats, cycles = [], []
    gather_bytes = 0
    for w, cyc, x in layers:
        ws = cyc.sel_cap
        pad = (w.R * ws,) + tuple(w.K.shape[1:])
        K2 = torch.cat([w.K, torch.zeros(pad, dtype=w.K.dtype, device=dev)])
        V2 = torch.cat([w.V, torch.zeros(pad, dtype=w.V.dtype, device=dev)])
        pool2 = kap.KVPool(K2, V2, w.Hq, torch.zeros(K2.shape[0], w.Hkv, w.d, dtype=torch.float32, device=dev))
        kap.kap_build_summaries(pool2, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
        tmp = kap.View.empty(w.R, cyc.rows, cyc.view_cap, dev)
        mats.append((pool2, kap.PageMap(w.block_table, w.ctx_len), cyc.view, w.num_pages, ws, tmp))
        c2 = kap.DecodeCycle(pool2, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q,
                             kap.rope_inv_freq(w.d, w.theta, dev), policy=cyc.policy, workspace_pages=(w.num_pages, ws))
        c2.plan(x["q_route"])
        cycles.append((c2, x))
        ns = cyc.n_sel.cpu().numpy().astype(np.int64)
        gather_bytes += int(ns.sum()) * 2 * PAGE * w.d * 2 * 2   # K and V chunks, read once and written once

    def run_mat():
        for pool2, pmap, view, first, ws, tmp in mats:
            kap.kap_materialize_view(pool2, pmap, view, first, ws, out_view=tmp)

    def run_prop():
        for c2, x in cycles:
            c2.propose_step(0, x["q_prop"][0], x["k_prop"][0], x["v_prop"][0], settled=True)

    out = {}
    for name, fn in (("gather", run_mat), ("propose", run_prop)):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        n = max(3, min(steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) * 1e3 / (n * len(layers))
    gb = gather_bytes / len(layers)
    return {"gather_us_per_layer": out["gather"], "gather_bytes_per_layer": gb,
            "gather_gbs": gb / (out["gather"] * 1e-6) / 1e9,
            "gather_pct_of_roofline": 100 * gb / (out["gather"] * 1e-6) / 1e9 / hbm_peak,
            "propose_us_per_launch": out["propose"],
            "note": "bytes = selected K+V read and written once; proposal = step 0 over the materialised views"}


# ------------------------------------------------------------------------------- tolerant acceptance, commit
ACCEPT_VOCAB = 128256   # Llama-3 vocabulary


def time_accept(layers, steps: int, hbm_peak: float, dev):
    """Times kap_accept_commit (KAP paper, verifier: Top-3 tolerant acceptance of the carry + k proposal window, next
    carry, committed length) on fp32 logits of the carry + 4 proposals of every request, three distinct logit sets
    per layer so that the logits read per replay exceed L2."""
    import torch
    import selected_kv_sparse_gb300 as kap
    from workloads import make_verify_logits, make_workload
    w0 = layers[0][0]
    calls = []
    for li in range(len(layers)):
        for rep in range(3):
            wk = make_workload(CONFIG, device="cpu", scale=1 / 64, poison=False, n_q_override=w0.k_prop + 1)
            lg, tok, off = make_verify_logits(wk, ACCEPT_VOCAB, device=dev, seed_offset=li * 3 + rep)
            R, rows = wk.R, int(off[-1].item())
            start = torch.full((R,), 32768, dtype=torch.int32, device=dev)
            outs = [torch.zeros(R, dtype=torch.int32, device=dev) for _ in range(3)]
            ws = torch.zeros(kap.kap_accept_workspace_size(R, rows, ACCEPT_VOCAB), dtype=torch.uint8, device=dev)
            calls.append((lg, off, tok, start, outs, ws))

    def run():
        for lg, off, tok, start, (acc, car, sl), ws in calls:
            kap.kap_accept_commit(lg, off, tok, 3, acc, car, ws, start_pos=start, seq_len_out=sl)
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    n = max(3, min(steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (n * len(calls))
    b = calls[0][0].numel() * 4
    acc_rate = float(torch.stack([c[4][0] for c in calls]).float().mean()) / w0.k_prop
    return {"us_per_call": us, "bytes_per_call": b, "gbs": b / (us * 1e-6) / 1e9,
            "pct_of_roofline": 100 * b / (us * 1e-6) / 1e9 / hbm_peak, "vocab": ACCEPT_VOCAB, "top_n": 3,
            "window": f"carry + {w0.k_prop} proposals x {w0.R} requests, fp32 logits",
            "acceptance_rate": acc_rate, "l2": f"{len(calls)} distinct logit sets, "
                                              f"{len(calls) * b / 1e6:.0f} MB per replay"}


# ------------------------------------------------------------------------------------ the other workloads
def policy_of(w):
    """Access policy of workload w: its A/R/K split (one for all requests, or one per request), per-KV-head or
    shared selection, and the selection capacity."""
    import selected_kv_sparse_gb300 as kap
    a, r, k = (int(x) for x in w.ark[0].tolist())
    same = bool((w.ark == w.ark[0]).all())
    return kap.AccessPolicy(a, r, k, w.per_kv_head, w.sel_cap(), None if same else w.ark.contiguous())


def time_workload(name: str, layers_n: int, steps: int, warmup: int, hbm_peak: float, dev, **kw):
    """One decode cycle of workload `name` per layer (plan, every proposal step fused with its append, window
    append, verification) over `layers_n` layer replicas, each phase one CUDA graph over the layers, timed with
    CUDA events between replays. Returns per-launch times, algorithmic bytes, GB/s and the fraction of the HBM
    roofline of the proposal and verification launches, the cycle time and the steps per second."""
    import torch
    import selected_kv_sparse_gb300 as kap
    from workloads import make_workload
    layers = []
    for l in range(layers_n):
        w = make_workload(name, device=dev, seed_offset=300 + l, poison=False, **kw)
        pool = kap.KVPool(w.K, w.V, w.Hq, torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev))
        kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
        pol = policy_of(w)
        cyc = kap.DecodeCycle(pool, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q,
                              kap.rope_inv_freq(w.d, w.theta, dev), policy=pol, spans=w.spans,
                              span_offsets=w.span_offsets, sel_cap=pol.cap)
        layers.append((w, cyc))
    k_prop = layers[0][0].k_prop
    phases = [("plan", lambda: [c.plan(w.q_route) for w, c in layers])]
    for i in range(k_prop):
        phases.append((f"prop{i}", lambda i=i: [c.propose_step(i, w.q_prop[i], w.k_new_prop[i], w.v_new_prop[i],
                                                               settled=True) for w, c in layers]))
    phases.append(("vapp", lambda: [c.append_window(w.q_ver, w.k_new_ver, w.v_new_ver) for w, c in layers]))
    phases.append(("ver", lambda: [c.verify(w.q_ver) for w, c in layers]))
    for _, fn in phases:
        fn()
    torch.cuda.synchronize()
    graphs = []
    for nm, fn in phases:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append((nm, g))
    for _ in range(warmup):
        for _, g in graphs:
            g.replay()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)] for _ in range(steps)]
    for s_ in range(steps):
        evs[s_][0].record()
        for j, (_, g) in enumerate(graphs):
            g.replay()
            evs[s_][j + 1].record()
    torch.cuda.synchronize()
    ph = {nm: sum(evs[s_][j].elapsed_time(evs[s_][j + 1]) for s_ in range(steps)) / steps
          for j, (nm, _) in enumerate(graphs)}
    by = [step_bytes(w, c, c.sel_ids, c.n_sel) for w, c in layers]
    L = layers_n
    b_prop = sum(sum(b["propose"]) for b in by) / (k_prop * L)
    b_ver = sum(b["verify"] for b in by) / L
    b_score = sum(b["score"] for b in by) / L
    t_prop = sum(ph[f"prop{i}"] for i in range(k_prop)) / (k_prop * L) * 1e-3   # s per launch
    t_ver = ph["ver"] / L * 1e-3
    t_cycle = sum(ph.values()) / L * 1e-3
    b_cycle = sum(b["score"] + sum(b["propose"]) + b["verify"] + b["append"] for b in by) / L
    w0 = layers[0][0]
    s_frac = [float(b["propose"][0]) for b in by]
    out = {
        "layers": L, "requests": w0.R, "proposal_steps_per_cycle": k_prop,
        "propose": {"us_per_launch": t_prop * 1e6, "bytes_per_launch": b_prop, "gbs": b_prop / t_prop / 1e9,
                    "pct_of_roofline": 100 * b_prop / t_prop / 1e9 / hbm_peak, "steps_per_s": 1.0 / t_prop},
        "verify": {"us_per_launch": t_ver * 1e6, "bytes_per_launch": b_ver, "gbs": b_ver / t_ver / 1e9,
                   "pct_of_roofline": 100 * b_ver / t_ver / 1e9 / hbm_peak, "steps_per_s": 1.0 / t_ver},
        "plan_us_per_layer": ph["plan"] / L * 1e3, "score_bytes_per_layer": b_score,
        "window_append_us_per_layer": ph["vapp"] / L * 1e3,
        "cycle": {"us_per_layer": t_cycle * 1e6, "bytes_per_layer": b_cycle, "gbs": b_cycle / t_cycle / 1e9,
                  "pct_of_roofline": 100 * b_cycle / t_cycle / 1e9 / hbm_peak, "cycles_per_s": 1.0 / t_cycle},
        "selected_fraction": b_prop / max(1.0, b_ver),
        "steps": steps, "warmup": warmup,
    }
    del layers, graphs, phases, by, s_frac
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------------------------------ arenas
class Arena:
    """One contiguous device buffer holding, for each of `copies` layers, tensors of the given (name, shape, dtype);
    each tensor starts on a 256-byte boundary."""

    def __init__(self, specs, copies, device):
        import torch
        self.specs = specs
        self.offsets = []
        off = 0
        for _ in range(copies):
            lay = {}
            for name, shape, dtype in specs:
                n = 1
                for x in shape:
                    n *= int(x)
                nbytes = n * torch.tensor([], dtype=dtype).element_size()
                lay[name] = (off, nbytes)
                off += (nbytes + 255) // 256 * 256
            self.offsets.append(lay)
        self.buf = torch.zeros(off, dtype=torch.uint8, device=device)

    def views(self, copy):
        out = {}
        for name, shape, dtype in self.specs:
            off, nbytes = self.offsets[copy][name]
            out[name] = self.buf[off:off + nbytes].view(dtype).view(shape)
        return out


# ------------------------------------------------------------------------------------------ recorded counters
KERNEL_SOURCES = {"verify_tc_kernel": ["k_verify.cu", "kap_device.cuh"],
                  "propose_kernel": ["k_propose.cu", "kap_device.cuh"]}


def kernel_source_hash(kernel: str) -> str:
    """SHA-256 of the kernel's sources with comments and blank space removed (a comment edit keeps the record)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "selected_kv_sparse_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def recorded_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the ncu capture summarised in profiles/, or None when
    no capture exists or the kernel's source has changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path))[kernel]
        if rec.get("source_sha256") != kernel_source_hash(kernel):
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------------------------------------ oracle arm
def oracle_sample(w_cpu, nthreads: int, r: int = 0):
    """Runs the oracle on one request of one layer for one full cycle of workload w_cpu (summaries, scores and A/R/K
    top-K per KV head or shared, or span selection; every proposal step; the verify window); returns (seconds,
    algorithmic bytes)."""
    import numpy as np
    import oracle
    bt = w_cpu.block_table.numpy()
    ctx = w_cpu.ctx_len.numpy()
    seq0 = w_cpu.seq_len0.numpy()
    npg = (int(ctx[r]) + max(w_cpu.k_prop, int(w_cpu.n_q[r])) + PAGE - 1) // PAGE
    pages = bt[r, :npg]
    K = w_cpu.K[pages].float().numpy()
    V = w_cpu.V[pages].float().numpy()
    lbt = np.arange(npg, dtype=np.int32)[None]
    lctx, lseq = ctx[r:r + 1], seq0[r:r + 1]
    qr = w_cpu.q_route[r:r + 1].float().numpy()
    a, rr, k = (int(x) for x in w_cpu.ark[r].tolist())
    N = (int(lctx[0]) + PAGE - 1) // PAGE
    rows = w_cpu.Hkv if w_cpu.per_kv_head else 1
    t0 = time.perf_counter()
    S = oracle.build_summaries(K, lbt, lctx)
    if w_cpu.spans is not None:
        so = w_cpu.span_offsets.numpy()
        sels = [oracle.select_spans(N, w_cpu.spans.numpy()[so[r]:so[r + 1]], a, rr)]
    else:
        sc, _ = oracle.scores(qr, S, lbt, lctx, per_head=w_cpu.per_kv_head)
        sels = [oracle.topk_ark(sc[0, v], N, a, rr, k) for v in range(rows)]
    cap = max(len(x) for x in sels)
    sel = np.zeros((1, rows, cap), np.int32)
    nsel = np.zeros((1, rows), np.int32)
    for v, x in enumerate(sels):
        sel[0, v, :len(x)] = x
        nsel[0, v] = len(x)
    for i in range(w_cpu.k_prop):
        q = w_cpu.q_prop[i, r:r + 1].float().numpy()
        oracle.attn_propose(q, K, V, lbt, lctx, lseq + i + 1, sel, nsel, nthreads=nthreads)
    nq = int(w_cpu.n_q[r])
    qv = w_cpu.q_ver[int(w_cpu.q_offsets[r]):int(w_cpu.q_offsets[r]) + nq].float().numpy()
    oracle.attn_verify(qv, K, V, lbt, np.array([0, nq], np.int32), lseq, nthreads=nthreads)
    dt = time.perf_counter() - t0
    kv_tok = w_cpu.d * 2 * 2
    prop_bytes = 0
    for i in range(w_cpu.k_prop):
        for h in range(w_cpu.Hkv):
            v = 0 if rows == 1 else h
            p = sel[0, v, :nsel[0, v]].astype(np.int64)
            prop_bytes += int((np.minimum(PAGE, int(lctx[0]) - PAGE * p).clip(min=0).sum() + i + 1) * kv_tok)
    ver_bytes = (int(lseq[0]) + nq) * w_cpu.Hkv * kv_tok
    score_bytes = N * w_cpu.Hkv * w_cpu.d * 4 if w_cpu.spans is None else 0
    return dt, prop_bytes + ver_bytes + score_bytes


def oracle_workloads(nthreads: int, budget_s: float = 3.0):
    """The oracle's time for one request-cycle of the long-context, EarlySelectKV (batch 1, one step) and mixed
    workloads at their stated sizes, each repeated over requests until `budget_s` seconds are spent."""
    from workloads import make_workload
    out = {}
    # the mixed batch's requests are timed on a batch of 4 drawn the same way, in a pool of just their pages
    for name, kw in (("long", {}), ("early", dict(batch=1)), ("mixed", dict(batch=4, pool_min_override=0))):
        w = make_workload(name, device="cpu", poison=False, **kw)
        dt = b = 0.0
        n = 0
        while dt < budget_s:
            t_, b_ = oracle_sample(w, nthreads, r=n % w.R)
            dt += t_
            b += b_
            n += 1
        out[name] = {"ms_per_request_cycle": dt / n * 1e3, "gbs": b / dt / 1e9, "cycles": n, "cores": nthreads}
        del w
    return out


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import torch
    import oracle
    from workloads import make_workload
    oracle.build()
    nthreads = oracle.hardware_threads()
    w = make_workload(CONFIG, device="cpu", poison=False)
    for _ in range(args.warmup):
        oracle_sample(w, nthreads)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, b = oracle_sample(w, nthreads)
        times.append(dt)
        nbytes = b
    tot = sum(times)
    val = nbytes * args.steps / tot / 1e9
    sample = (f"one request of one layer per step: block-mean summaries, fixed-order scores and A1R2K125 top-K for "
              f"8 KV heads, 4 proposal attentions and one verify window of 4 over the 32772-token context, fp64")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": nthreads, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------------------------- GPU arm
def run_kap(args, world, rank, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    import selected_kv_sparse_gb300 as kap
    from workloads import make_workload
    kap.load()

    L = args.layers
    # All layers' inputs live in one device buffer and all outputs in another (views per layer), so the
    # end-to-end step moves each direction with a single copy.
    layers = []
    out_arena = None
    for l in range(L):
        w = make_workload(CONFIG, device=dev, seed_offset=rank * 1000 + l, poison=False)
        ksum = torch.zeros(w.num_pages, w.Hkv, w.d, dtype=torch.float32, device=dev)
        pool = kap.KVPool(w.K, w.V, w.Hq, ksum)
        kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
        a, r, k = (int(x) for x in w.ark[0].tolist())
        pol = kap.AccessPolicy(a, r, k, True, w.sel_cap())
        if out_arena is None:
            probe = kap.DecodeCycle(pool, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q,
                                    kap.rope_inv_freq(w.d, w.theta, dev), policy=pol, fused=not args.unfused)
            out_arena = Arena([(n, sh, dt) for n, (sh, dt) in probe.output_shapes().items()], L, dev)
            del probe
        cyc = kap.DecodeCycle(pool, w.block_table, w.ctx_len, w.seq_len0, w.k_prop, w.n_q,
                              kap.rope_inv_freq(w.d, w.theta, dev), policy=pol, fused=not args.unfused,
                              outputs=out_arena.views(l), overlap=not args.no_overlap)
        ins = dict(q_route=w.q_route, q_prop=w.q_prop, k_prop=w.k_new_prop, v_prop=w.v_new_prop, q_ver=w.q_ver,
                   k_ver=w.k_new_ver, v_ver=w.v_new_ver)
        layers.append((w, cyc, ins))
    in_arena = Arena([(n, tuple(t.shape), t.dtype) for n, t in layers[0][2].items()], L, dev)
    for l, (_, _, x) in enumerate(layers):
        views = in_arena.views(l)
        for n in list(x):
            views[n].copy_(x[n])
            x[n] = views[n]
    k_prop = layers[0][0].k_prop

    # Each phase runs every layer's call and is replayed as its own CUDA graph, so the plan graph that wrote the
    # views has completed before any proposal launch, and within a proposal graph the kernel ahead of a layer's
    # launch belongs to another layer: every proposal call may treat its view as settled.
    st = None if args.no_overlap else True
    phases = [("plan", lambda: [c.plan(x["q_route"]) for _, c, x in layers])]
    for i in range(k_prop):
        if args.unfused:
            phases.append((f"app{i}", lambda i=i: [c.append_step(i, x["q_prop"][i], x["k_prop"][i], x["v_prop"][i])
                                                    for _, c, x in layers]))
            phases.append((f"prop{i}", lambda i=i: [c.propose(i, x["q_prop"][i], settled=st) for _, c, x in layers]))
        else:   # the step's KV append runs inside the proposal kernel
            phases.append((f"prop{i}", lambda i=i: [c.propose_step(i, x["q_prop"][i], x["k_prop"][i], x["v_prop"][i],
                                                                   settled=st) for _, c, x in layers]))
    phases.append(("vapp", lambda: [c.append_window(x["q_ver"], x["k_ver"], x["v_ver"]) for _, c, x in layers]))
    phases.append(("ver", lambda: [c.verify(x["q_ver"]) for _, c, x in layers]))

    # eager pass (sets kernel attributes, caches tensor maps), then one CUDA graph per phase
    for _, fn in phases:
        fn()
    torch.cuda.synchronize()
    graphs = []
    for name, fn in phases:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append((name, g))
    torch.cuda.synchronize()
    launches_per_step = sum(c.launches_per_cycle() for _, c, _ in layers)

    # algorithmic bytes (selection is fixed across cycles: the routing query is not modified by a cycle)
    by = [step_bytes(w, c, c.sel_ids, c.n_sel) for w, c, _ in layers]
    b_score = sum(b["score"] for b in by)
    b_prop = [sum(b["propose"][i] for b in by) for i in range(k_prop)]
    b_ver = sum(b["verify"] for b in by)
    b_app = sum(b["append"] for b in by)
    b_step = b_score + sum(b_prop) + b_ver + b_app
    ws_bytes = sum(x.K.numel() * 2 * 2 for x, _, _ in layers)

    def replay_step(evs=None):
        if evs is not None:
            evs[0].record()
        for j, (_, g) in enumerate(graphs):
            g.replay()
            if evs is not None:
                evs[j + 1].record()

    for _ in range(args.warmup):
        replay_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)] for _ in range(K)]
    sampler = ClockSampler(local, args.clock_log)
    sampler.start()
    time.sleep(0.05)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record()
    for s in range(K):
        replay_step(evs[s])
    t_end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    total_ms_local = t_start.elapsed_time(t_end)
    phase_ms = {name: 0.0 for name, _ in graphs}
    for s in range(K):
        for j, (name, _) in enumerate(graphs):
            phase_ms[name] += evs[s][j].elapsed_time(evs[s][j + 1])
    total_ms = reduce_max(total_ms_local, dist)
    ms_step = total_ms / K
    bytes_all = reduce_sum(float(b_step), dist)
    value = bytes_all / (ms_step * 1e-3) / 1e9

    hbm_peak, peak_kind = measured_peaks()
    ver_launch_ms = phase_ms["ver"] / (K * L)
    prop_launch_ms = sum(phase_ms[f"prop{i}"] for i in range(k_prop)) / (K * k_prop * L)
    ver_bytes_launch = b_ver / L
    prop_bytes_launch = sum(b_prop) / (k_prop * L)
    ver_gbs = ver_bytes_launch / (ver_launch_ms * 1e-3) / 1e9
    prop_gbs = prop_bytes_launch / (prop_launch_ms * 1e-3) / 1e9
    plan_ms = phase_ms["plan"] / (K * L)
    traffic = recorded_traffic("verify_tc_kernel")

    # end to end: inputs from pinned host memory, results back, through the same calls
    e2e = None
    if not args.no_e2e:
        # every layer's inputs from one pinned host buffer, every output back into another: one copy each way
        host_in = in_arena.buf.cpu().pin_memory()
        host_out = torch.empty(out_arena.buf.shape, dtype=torch.uint8, pin_memory=True)
        h2d = host_in.numel()
        d2h = host_out.numel()
        n_e2e = max(3, min(K, 50))

        def e2e_step():
            in_arena.buf.copy_(host_in, non_blocking=True)
            replay_step()
            host_out.copy_(out_arena.buf, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        for _ in range(2):
            e2e_step()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n_e2e):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        e_ms = reduce_max(e0.elapsed_time(e1), dist) / n_e2e
        e2e = {"value": bytes_all / (e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e, "ms_per_step": e_ms}

    prior = None if args.no_prior else time_prior(layers, K, hbm_peak, dev)
    accept = None if args.no_accept else time_accept(layers, K, hbm_peak, dev)
    mat = None if args.no_materialize else time_materialize(layers, K, hbm_peak, dev)
    side = None if args.no_side_flow else time_side_flow(K, dev, hbm_peak)
    loop = None if args.no_decode_loop else time_decode_loop(dev, hbm_peak)
    other = None
    if not args.no_configs:
        nst = max(3, min(K, 20))
        other = {
            "long": dict(time_workload("long", 8, nst, 3, hbm_peak, dev),
                         workload="GraphSpec-like long context: 1 request x 131072 tokens (8192 pages), Hq 40, Hkv 8, "
                                  "d 128, 451-page evidence-span view (s = 5.5%) shared by the KV heads, 8 proposal "
                                  "steps + verify window 8 per cycle, 8 layer replicas"),
            "mixed": dict(time_workload("mixed", 1, nst, 3, hbm_peak, dev),
                          workload="mixed serving batch: 32 requests, prompts log-uniform in 4K-128K tokens, s in "
                                   "{2, 5.5, 10, 25}%, splits A1R2/A4R4/A0R0, 1 proposal launch for all requests + 1 "
                                   "verify launch with windows {2, 4, 8}, shared 2^20-page pool (64 GiB)"),
        }

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        nth = oracle.hardware_threads()
        w_cpu = make_workload(CONFIG, device="cpu", poison=False)
        dt = b = 0.0
        n_cyc = 0
        while dt < 10.0:     # about ten seconds of oracle work, cycling over the requests
            t_, b_ = oracle_sample(w_cpu, nth, r=n_cyc % w_cpu.R)
            dt += t_
            b += b_
            n_cyc += 1
        # the same cycles on one thread (the oracle's attention is parallel over (row, head) units)
        dt1 = b1 = 0.0
        n1 = 0
        while dt1 < 6.0:
            t_, b_ = oracle_sample(w_cpu, 1, r=n1 % w_cpu.R)
            dt1 += t_
            b1 += b_
            n1 += 1
        per_workload = oracle_workloads(nth)
        cpu = {"value": b / dt / 1e9, "unit": "GB/s", "cores": nth, "kind": "oracle",
               "other_workloads": per_workload,
               "sample": f"{n_cyc} full cycles, each one request of one layer (summaries, fixed-order scores, "
                         f"A1R2K125 top-K, 4 proposals, verify window 4) in fp64: {dt:.1f} s",
               "single_thread": {"value": b1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                                 "sample": f"{n1} of the same cycles on one thread: {dt1:.1f} s"},
               "ms_per_request_layer_cycle": {"all_cores": dt / n_cyc * 1e3, "one_thread": dt1 / n1 * 1e3}}

    dev_err = kap.kap_device_error()   # nonzero: a kernel met a bad page, length or timed-out wait
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers_per_step": L, "parallelism": "replicas" if world > 1 else "1 GPU",
                       "calls": "separate" if args.unfused else "fused",
                       "proposal_overlap": not args.no_overlap,
                       "l2": f"inputs larger than L2: {ws_bytes / 2**30:.1f} GiB of KV per rank, "
                             f"{b_step / 2**30:.2f} GiB read per step"},
            "pct_of_hbm_roofline": 100.0 * value / (hbm_peak * world),
            "propose": {"gbs": prop_gbs, "pct_of_roofline": 100 * prop_gbs / hbm_peak,
                        "us_per_launch": prop_launch_ms * 1e3, "bytes_per_launch": prop_bytes_launch,
                        "steps_per_s": 1e3 / (prop_launch_ms)},
            "verify": {"gbs": ver_gbs, "pct_of_roofline": 100 * ver_gbs / hbm_peak,
                       "us_per_launch": ver_launch_ms * 1e3, "bytes_per_launch": ver_bytes_launch,
                       "steps_per_s": 1e3 / ver_launch_ms},
            "plan_us_per_layer": plan_ms * 1e3,
            "plan": {"us_per_layer": plan_ms * 1e3, "score_bytes_per_layer": b_score / L,
                     "gbs": (b_score / L) / (plan_ms * 1e-3) / 1e9,
                     "pct_of_roofline": 100 * (b_score / L) / (plan_ms * 1e-3) / 1e9 / hbm_peak,
                     "note": "scoring bytes (one fp32 summary per prompt page and KV head) over the whole plan "
                             "phase: scores, top-K and view"},
            "prior_topk": prior,
            "accept_commit": accept,
            "materialize": mat,
            "early_side_flow": side,
            "early_decode_loop": loop,
            "workloads": other,
            "phase_ms_per_step": {k2: v / K for k2, v in phase_ms.items()},
            "roofline": {"bound": "hbm", "kernel": "verify_tc_kernel", "achieved": ver_gbs, "peak": hbm_peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": ver_gbs / hbm_peak, "traffic": traffic},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * K,
            "device_error": dev_err,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_kap(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
