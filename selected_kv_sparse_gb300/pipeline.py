"""One proposal/verification cycle of the selected-KV decode loop over one attention layer, on the library calls.

KAP paper, executor and verifier: the plan (selection, compact view, slot mapping) is compiled once per cycle;
each of the k proposal steps appends the step's token KV (RoPE at its logical position) and runs q = 1 attention
over the compact view, in one fused call (kap_append_propose) or as kap_append_kv + kap_attn_propose; the verifier
appends the window's KV into the full-context slots and runs causal q = n attention over the full block table.
Every buffer is allocated here, once; the calls themselves allocate nothing, so a cycle can be captured in a CUDA
graph.

With overlap (the default), a proposal call that does not directly follow the plan marks the view as settled: its
kernel then scans the view and starts streaming the selected prompt pages while the previous kernel finishes. The
cycle tracks its own launches for this; a caller that launches kernels writing the view, the page map or prompt
tokens on the same stream between the cycle's calls must pass overlap=False.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding as kb

PAGE = 16


class DecodeCycle:
    def __init__(self, pool: kb.KVPool, block_table: torch.Tensor, ctx_len: torch.Tensor, seq_len0: torch.Tensor,
                 k_prop: int, n_q: torch.Tensor, inv_freq: torch.Tensor, policy: Optional[kb.AccessPolicy] = None,
                 spans: Optional[torch.Tensor] = None, span_offsets: Optional[torch.Tensor] = None,
                 sel_cap: Optional[int] = None, s_max: float = 1.0, fused: bool = True,
                 outputs: Optional[dict] = None, overlap: bool = True,
                 workspace_pages: Optional[tuple] = None):
        dev = block_table.device
        self.fused = bool(fused)
        # (first pool page, pages per request) of a materialised compact workspace, or None for the zero-copy view
        self.workspace_pages = tuple(workspace_pages) if workspace_pages is not None else None
        self.overlap = bool(overlap)
        self._view_fresh = True  # the last launch of this cycle wrote the view (or none has run yet)
        self.pool = pool
        self.R = int(block_table.shape[0])
        self.Hq = pool.num_q_heads
        self.Hkv = int(pool.k_pages.shape[1])
        self.d = int(pool.k_pages.shape[3])
        self.k_prop = int(k_prop)
        self.inv_freq = inv_freq
        self.policy = policy
        self.spans, self.span_offsets = spans, span_offsets
        if policy is None or (spans is None and policy is None):
            raise ValueError("a policy is required")
        self.rows = self.Hkv if (policy.per_kv_head and spans is None) else 1
        n_q_host = [int(x) for x in n_q.cpu().tolist()]
        self.max_q = max(n_q_host)
        self.total_q = sum(n_q_host)
        self.horizon = max(self.k_prop, self.max_q)
        self.sel_cap = int(sel_cap if sel_cap is not None else policy.cap)
        self.view_cap = self.sel_cap + (self.horizon + PAGE - 1) // PAGE + 1
        self.s_max = s_max
        i32 = dict(dtype=torch.int32, device=dev)
        # page maps: the plan's (committed length) and one per proposal step (query at seq_len0 + i)
        self.map_plan = kb.PageMap(block_table, ctx_len, seq_len0)
        self.seq_steps = [(seq_len0 + i + 1).to(torch.int32).contiguous() for i in range(self.k_prop)]
        self.map_steps = [kb.PageMap(block_table, ctx_len, s) for s in self.seq_steps]
        self.map_full = kb.PageMap(block_table, ctx_len, seq_len0)
        # selection, view, fallback flags
        self.sel_ids = torch.zeros(self.R, self.rows, self.sel_cap, **i32)
        self.n_sel = torch.zeros(self.R, self.rows, **i32)
        self.view = kb.View.empty(self.R, self.rows, self.view_cap, dev)
        self.fallback = torch.zeros(self.R, **i32)
        # slot mappings: the horizon tokens [R][horizon] come with the view; the verify window [total_q] reuses
        # them when every window spans exactly the horizon, else gets its own mapping
        self.slots_prop = torch.zeros(self.R * self.horizon, dtype=torch.int64, device=dev)
        self.pos_prop = torch.zeros(self.R * self.horizon, **i32)
        self.window_is_horizon = all(n == self.horizon for n in n_q_host)
        q_off = torch.zeros(self.R + 1, dtype=torch.int32)
        q_off[1:] = torch.cumsum(torch.tensor(n_q_host, dtype=torch.int32), 0)
        self.q_offsets = q_off.to(dev)
        self.q_start = seq_len0.to(torch.int32).contiguous()
        if self.window_is_horizon:
            self.slots_ver, self.pos_ver = self.slots_prop, self.pos_prop
        else:
            self.slots_ver = torch.zeros(self.total_q, dtype=torch.int64, device=dev)
            self.pos_ver = torch.zeros(self.total_q, **i32)
        self.vpol = kb.VerifyPolicy(self.q_offsets, self.q_start, self.max_q, self.total_q)
        # workspaces (zero-filled once)
        mp = int(block_table.shape[1])
        self.ws_score = kb.workspace(kb.kap_score_workspace_size(self.R, self.rows, mp), dev)
        self.ws_prop = kb.workspace(kb.kap_propose_workspace_size(self.R, self.Hkv, self.Hq, self.d), dev)
        self.ws_ver = kb.workspace(kb.kap_verify_workspace_size(self.R, self.Hkv, self.Hq, self.d, self.max_q), dev)
        # outputs (caller-provided tensors of these shapes may be passed in `outputs`, e.g. views of one buffer)
        shapes = self.output_shapes()
        outputs = outputs or {}
        for name, (shape, odt) in shapes.items():
            t = outputs.get(name)
            if t is None:
                t = torch.empty(shape, dtype=odt, device=dev)
            elif tuple(t.shape) != tuple(shape) or t.dtype != odt or not t.is_contiguous():
                raise ValueError(f"output {name} must be a contiguous {odt} tensor of shape {tuple(shape)}")
            setattr(self, name, t)

    def output_shapes(self) -> dict:
        """Shapes and dtypes of the cycle's outputs: proposal outputs and LSEs per step, verify outputs and LSEs."""
        dt = self.pool.dtype
        return {"o_prop": ((self.k_prop, self.R, self.Hq, self.d), dt),
                "lse_prop": ((self.k_prop, self.R, self.Hq), torch.float32),
                "o_ver": ((self.total_q, self.Hq, self.d), dt),
                "lse_ver": ((self.total_q, self.Hq), torch.float32)}

    # -------------------------------------------------------------------------------------------------- phases
    def plan(self, q_route: torch.Tensor, stream=None):
        """Selection (scores + A/R/K top-K, or spans), compact view and both slot mappings. Fused, score selection
        and view compilation are one call (kap_score_topk_view)."""
        if self.spans is not None:
            kb.kap_select_spans(self.map_plan, self.spans, self.span_offsets, self.policy, self.sel_ids, self.n_sel,
                                stream)
        elif self.fused:
            kb.kap_score_topk_view(self.pool, self.map_plan, q_route, self.policy, self.sel_ids, self.n_sel,
                                   self.ws_score, self.horizon, self.view, self.fallback, self.s_max, self.slots_prop,
                                   self.pos_prop, stream)
        else:
            kb.kap_score_topk(self.pool, self.map_plan, q_route, self.policy, self.sel_ids, self.n_sel, self.ws_score,
                              stream)
        if self.spans is not None or not self.fused:
            kb.kap_compile_view(self.map_plan, self.sel_ids, self.n_sel, self.horizon, self.view, self.fallback,
                                self.s_max, self.slots_prop, self.pos_prop, stream)
        if not self.window_is_horizon:
            kb.kap_slot_mapping(self.map_plan, self.q_offsets, self.q_start, self.slots_ver, self.pos_ver, stream)
        if self.workspace_pages is not None:   # copy the selected pages into the workspace, view rewritten in place
            kb.kap_materialize_view(self.pool, self.map_plan, self.view, self.workspace_pages[0],
                                    self.workspace_pages[1],
                                    fallback=self.fallback, stream=stream)
        self._view_fresh = True

    def _settled(self, override: Optional[bool]) -> bool:
        """Whether the next launch may treat the view as settled (override: the caller knows its launch order); the
        launch itself makes the view settled for the one after."""
        s = (self.overlap and not self._view_fresh) if override is None else bool(override)
        self._view_fresh = False
        return s

    def append_step(self, i: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Proposal step i, first half: the step token's KV at its logical position (q rotated in place)."""
        kb.kap_append_kv(self.pool, k_new, v_new, q, self.pos_prop[i:], self.slots_prop[i:], self.inv_freq,
                         num_tokens=self.R, tok_stride=self.horizon, stream=stream)
        self._view_fresh = False

    def propose(self, i: int, q: torch.Tensor, stream=None, settled: Optional[bool] = None):
        """Proposal step i, second half: q = 1 attention over the compact view."""
        kb.kap_attn_propose(self.pool, self.map_steps[i], self.view, q, self.o_prop[i], self.lse_prop[i], self.ws_prop,
                            stream, settled=self._settled(settled))

    def propose_step(self, i: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None,
                     settled: Optional[bool] = None):
        """Proposal step i: append the step token's KV and attend. Fused, q is read before RoPE and left as it is;
        unfused, kap_append_kv rotates q in place first. settled: None decides from this cycle's own launches; True
        is the caller's promise that the kernel launched just ahead of this one did not write the view, the page
        map or prompt tokens."""
        if self.fused:
            kb.kap_append_propose(self.pool, self.map_steps[i], self.view, q, k_new, v_new, self.inv_freq,
                                  self.o_prop[i], self.lse_prop[i], self.ws_prop, stream, settled=self._settled(settled))
        else:
            self.append_step(i, q, k_new, v_new, stream)
            self.propose(i, q, stream, settled)

    def append_window(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """The verify window's KV into the full-context slots (q rotated in place)."""
        kb.kap_append_kv(self.pool, k_new, v_new, q, self.pos_ver, self.slots_ver, self.inv_freq, stream=stream)
        self._view_fresh = False

    def verify(self, q: torch.Tensor, k_new: torch.Tensor = None, v_new: torch.Tensor = None, stream=None):
        """Causal attention of the window over the full table (after append_window when k_new/v_new are given)."""
        if k_new is not None:
            self.append_window(q, k_new, v_new, stream)
        kb.kap_attn_verify(self.pool, self.map_full, self.vpol, q, self.o_ver, self.lse_ver, self.ws_ver, stream)
        self._view_fresh = False

    def run(self, q_route, q_prop, k_new_prop, v_new_prop, q_ver, k_new_ver, v_new_ver, stream=None):
        self.plan(q_route, stream)
        for i in range(self.k_prop):
            self.propose_step(i, q_prop[i], k_new_prop[i], v_new_prop[i], stream)
        self.verify(q_ver, k_new_ver, v_new_ver, stream)

    def launches_per_cycle(self) -> int:
        """Kernel launches of one run(): selection and view (score + top-K with the view fused in; unfused score,
        top-K and view; or spans and view), a separate window slot mapping when the windows differ from the
        horizon, per step one fused kernel (or an append and a proposal kernel), then the window append and
        verification; plus the materialisation when a workspace is used."""
        sel_view = 2 if self.spans is not None else (2 if self.fused else 3)
        sel_view += 1 if self.workspace_pages is not None else 0
        slots = 0 if self.window_is_horizon else 1
        per_step = 1 if self.fused else 2
        return sel_view + slots + per_step * self.k_prop + 2


class SideFlowDecode:
    """EarlySelectKV side flow over a stack of layers: the routing of layer l + 1 (scores on a proxy query, top-K,
    compact view) runs on a second stream while layer l appends its token and attends on the main stream.

    EarlySelectKV page: selection stops waiting for the target layer's query; a proxy available earlier drives the
    routing, so its latency hides behind the attention of the layers before. Layer l's attention waits only for its
    own routing (an event); the routing of layer l + 1 waits for nothing of layer l. Every call allocates nothing,
    so a step can be captured in a CUDA graph (the side stream forks from and joins the capturing stream).
    `cycles` are one DecodeCycle per layer, each with one proposal step per decode step.
    """

    def __init__(self, cycles, side_stream: Optional[torch.cuda.Stream] = None):
        self.cycles = list(cycles)
        self.side = side_stream if side_stream is not None else torch.cuda.Stream(self.cycles[0].view.block_table.device)
        self.routed = [torch.cuda.Event() for _ in self.cycles]

    def step(self, q_route, q, k_new, v_new, overlap: bool = True):
        """One decode step over every layer: q_route[l] is layer l's proxy query, q[l], k_new[l], v_new[l] its
        step token's query, key and value. overlap=False runs routing and attention of each layer in turn on the
        current stream (the same calls, the same results)."""
        main = torch.cuda.current_stream()
        L = len(self.cycles)
        if not overlap:
            for l, c in enumerate(self.cycles):
                c.plan(q_route[l], main)
                c.propose_step(0, q[l], k_new[l], v_new[l], main)
            return
        self.side.wait_stream(main)  # the step's inputs are ready on the main stream
        with torch.cuda.stream(self.side):
            self.cycles[0].plan(q_route[0], self.side)
            self.routed[0].record(self.side)
        for l, c in enumerate(self.cycles):
            if l + 1 < L:   # next layer's routing goes out first, so that it runs while this layer attends
                with torch.cuda.stream(self.side):
                    self.cycles[l + 1].plan(q_route[l + 1], self.side)
                    self.routed[l + 1].record(self.side)
            main.wait_event(self.routed[l])
            # Not settled: the view comes from a kernel on the other stream. In a captured graph every incoming
            # edge of a dependent launch is programmatic, the one from the routing kernel included, so the proposal
            # may start before the routing has finished; it must read the view only after its dependency wait.
            c.propose_step(0, q[l], k_new[l], v_new[l], main, settled=False)
        main.wait_stream(self.side)


class DecodeLoop:
    """EarlySelectKV decode over `steps` generated tokens on one attention layer, on the library calls.

    EarlySelectKV page: every decode step routes (scores the K-summary cache on a proxy query, keeps the top pages)
    and then attends with the real query over the chosen pages only. Before step t the routing compiles the view at
    the committed length seq_len0 + t with a one-token horizon; step t then appends its token at position
    seq_len0 + t and attends over the selected prompt pages and every generated token (the view's tail grows by a
    page every 16 steps). Summaries cover prompt tokens only, so the generated tokens need no refresh.

    The lengths of every step are known ahead (one token per step), so each step has its own page map in device
    memory and nothing runs on the host between steps: a run of steps can be captured in one CUDA graph. plan() and
    propose_step() act on the current step; advance() moves to the next (the same interface as DecodeCycle's
    single-step use, so SideFlowDecode can run a stack of loops).
    """

    def __init__(self, pool: kb.KVPool, block_table: torch.Tensor, ctx_len: torch.Tensor, seq_len0: torch.Tensor,
                 steps: int, inv_freq: torch.Tensor, policy: kb.AccessPolicy, s_max: float = 1.0):
        dev = block_table.device
        self.pool, self.policy, self.inv_freq, self.s_max = pool, policy, inv_freq, s_max
        self.steps = int(steps)
        self.R = int(block_table.shape[0])
        self.Hq = pool.num_q_heads
        self.Hkv = int(pool.k_pages.shape[1])
        self.d = int(pool.k_pages.shape[3])
        self.rows = self.Hkv if policy.per_kv_head else 1
        self.sel_cap = int(policy.cap)
        self.view_cap = self.sel_cap + (self.steps + PAGE - 1) // PAGE + 2   # selected pages + every tail page
        ar = torch.arange(self.steps + 1, dtype=torch.int32, device=dev)
        self.lens = (seq_len0.to(torch.int32)[None, :] + ar[:, None]).contiguous()   # [steps + 1][R]
        self.maps = [kb.PageMap(block_table, ctx_len, self.lens[t]) for t in range(self.steps + 1)]
        i32 = dict(dtype=torch.int32, device=dev)
        self.sel_ids = torch.zeros(self.R, self.rows, self.sel_cap, **i32)
        self.n_sel = torch.zeros(self.R, self.rows, **i32)
        self.view = kb.View.empty(self.R, self.rows, self.view_cap, dev)
        self.fallback = torch.zeros(self.R, **i32)
        self.slots = torch.zeros(self.R, dtype=torch.int64, device=dev)
        self.pos = torch.zeros(self.R, **i32)
        mp = int(block_table.shape[1])
        self.ws_score = kb.workspace(kb.kap_score_workspace_size(self.R, self.rows, mp), dev)
        self.ws_prop = kb.workspace(kb.kap_propose_workspace_size(self.R, self.Hkv, self.Hq, self.d), dev)
        self.o = torch.empty(self.steps, self.R, self.Hq, self.d, dtype=pool.dtype, device=dev)
        self.lse = torch.empty(self.steps, self.R, self.Hq, dtype=torch.float32, device=dev)
        self.t = 0
        self._routed = False

    def plan(self, q_route: torch.Tensor, stream=None):
        """Routing of step t: scores on q_route [R][Hq][d], A/R/K top-K and the view at length seq_len0 + t."""
        kb.kap_score_topk_view(self.pool, self.maps[self.t], q_route, self.policy, self.sel_ids, self.n_sel,
                               self.ws_score, 1, self.view, self.fallback, self.s_max, self.slots, self.pos, stream)
        self._routed = True

    def propose_step(self, i: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, stream=None,
                     settled: Optional[bool] = None):
        """Step t: the token's K (RoPE at seq_len0 + t) and V into the pool, attention of q (before RoPE) over the
        view; outputs o[t], lse[t]. i is the step's index within a cycle and must be 0 (one token per step)."""
        if i != 0:
            raise ValueError("a decode step proposes one token")
        st = (not self._routed) if settled is None else bool(settled)
        kb.kap_append_propose(self.pool, self.maps[self.t + 1], self.view, q, k_new, v_new, self.inv_freq,
                              self.o[self.t], self.lse[self.t], self.ws_prop, stream, settled=st)
        self._routed = False

    def advance(self):
        if self.t + 1 > self.steps:
            raise ValueError("the loop has run all its steps")
        self.t += 1

    def reset(self):
        """Back to step 0 (a replayed loop writes the same tokens into the same slots)."""
        self.t = 0
        self._routed = False
