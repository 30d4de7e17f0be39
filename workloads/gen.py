"""Seeded generators for the five synthetic workloads of the selected-KV decode hot path.

Each configuration is named by what it is, with its sizes:
  tiny   - 1 request, Hq=8, Hkv=2, d=64, fp32, 1024-token prompt (64 pages in a 128-page pool), A1R2K5 per KV
           head, 2 needle pages, 1 proposal step, verify window 4.
  llama  - Llama-3-8B-shaped layer: 4 requests, Hq=32, Hkv=8, d=128, bf16, 32768-token prompts (2048 pages),
           A1R2K125 per KV head (s = 6.25%), 16 needle pages per request, 4 proposal steps, verify window 4.
  long   - 1 request, Hq=40, Hkv=8, d=128, bf16, 131072-token prompt (8192 pages); a shared view of 451 pages from
           30 evidence spans of 8-32 pages plus anchor page 0 and the last 4 pages; 8 proposal steps, verify 8.
  early  - EarlySelectKV-like: Hq=32, Hkv=8, d=128, bf16, 40960-token prompts (2560 pages), A0R0K8 per KV head
           (128-token budget), proxy query = query + N(0, 0.3^2); batch 1 or 8; one decode token per step.
  mixed  - 32 requests with prompt lengths log-uniform in 4K-128K tokens, retention s in {2, 5.5, 10, 25}%,
           splits A1R2 / A4R4 / A0R0, verify windows in {2, 4, 8}, 5 needles each, over a 2^20-page pool.

`scale` shrinks prompt lengths (and the mixed batch) while keeping every structural feature, so that the oracle
finishes in seconds; ragged prompt lengths (a partial last page) can be forced with `ragged=True`.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

PAGE = 16
SEED_BASE = 0x4B4150

CONFIGS = ("tiny", "llama", "long", "early", "mixed")


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    R: int
    Hq: int
    Hkv: int
    d: int
    num_pages: int
    K: torch.Tensor                 # [P][Hkv][16][d]
    V: torch.Tensor                 # [P][Hkv][16][d]
    block_table: torch.Tensor       # [R][max_pages] int32
    ctx_len: torch.Tensor           # [R] int32 prompt tokens
    seq_len0: torch.Tensor          # [R] int32 tokens present at the start of the cycle
    k_prop: int                     # proposal steps per cycle
    q_prop: torch.Tensor            # [k_prop][R][Hq][d] proposal queries
    q_route: torch.Tensor           # [R][Hq][d] routing query (the first proposal query, or a proxy of it)
    k_new_prop: torch.Tensor        # [k_prop][R][Hkv][d] keys of the proposed tokens (before RoPE)
    v_new_prop: torch.Tensor        # [k_prop][R][Hkv][d]
    n_q: torch.Tensor               # [R] int32 verify window per request
    q_offsets: torch.Tensor         # [R+1] int32
    q_ver: torch.Tensor             # [total_q][Hq][d] verify queries
    k_new_ver: torch.Tensor         # [total_q][Hkv][d] keys of the window tokens (before RoPE)
    v_new_ver: torch.Tensor         # [total_q][Hkv][d]
    ark: torch.Tensor               # [R][3] int32 anchor, recent, top-k per request
    per_kv_head: bool
    spans: Optional[torch.Tensor] = None        # [S][2] int32 token spans (first, length), span mode only
    span_offsets: Optional[torch.Tensor] = None  # [R+1] int32
    needles: List[List[int]] = field(default_factory=list)
    theta: float = 1.0e4
    sigma: float = 1.0
    # [k_prop][R][Hq][d] the routing query of every proposal step (early workload: each step's own noisy proxy of
    # its query, for a decode loop that re-routes at every step); step 0 equals q_route
    q_route_steps: Optional[torch.Tensor] = None

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_q(self) -> int:
        return int(self.n_q.max().item())

    @property
    def total_q(self) -> int:
        return int(self.q_offsets[-1].item())

    def sel_cap(self) -> int:
        a = self.ark.to(torch.int64)
        n = (self.ctx_len.to(torch.int64).cpu() + PAGE - 1) // PAGE
        if self.spans is not None:
            return int(n.max().item())
        return int(torch.minimum(n, (a[:, 0] + a[:, 1] + a[:, 2]).cpu()).max().item())


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, scale=1.0):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * scale


def _spans_long(g_cpu, n_pages: int, n_spans: int = 30, total: int = 446, lo: int = 8, hi: int = 32,
                a: int = 1, r: int = 4):
    """Evidence spans of the long-context workload: n_spans lengths in [lo, hi] adjusted to sum to `total`,
    placed non-overlapping and non-adjacent inside the middle pages [a, n_pages - r)."""
    lens = torch.randint(lo, hi + 1, (n_spans,), generator=g_cpu).tolist()
    while sum(lens) > total:
        i = max(range(n_spans), key=lambda j: (lens[j], -j))
        if lens[i] <= lo:
            break
        lens[i] -= 1
    while sum(lens) < total:
        i = min(range(n_spans), key=lambda j: (lens[j], j))
        if lens[i] >= hi:
            break
        lens[i] += 1
    mid_lo, mid_hi = a, n_pages - r
    free = (mid_hi - mid_lo) - sum(lens) - (n_spans - 1)
    if free < 0:
        raise ValueError("spans do not fit")
    cuts = sorted(torch.randint(0, free + 1, (n_spans,), generator=g_cpu).tolist())
    gaps = [cuts[0]] + [cuts[i] - cuts[i - 1] for i in range(1, n_spans)]
    spans = []
    p = mid_lo
    for i in range(n_spans):
        p += gaps[i] + (1 if i > 0 else 0)
        spans.append((p * PAGE, lens[i] * PAGE))
        p += lens[i]
    return spans


def make_workload(name: str, device="cpu", scale: float = 1.0, ragged: bool = False, seed_offset: int = 0,
                  batch: Optional[int] = None, poison: bool = True, n_q_override: Optional[int] = None,
                  k_prop_override: Optional[int] = None, pool_min_override: Optional[int] = None) -> Workload:
    """Builds one seeded workload on `device`.

    scale < 1 shortens every prompt (never below 64 tokens) and, for `mixed`, the batch, keeping the structure.
    pool_min_override replaces the workload's minimum pool size (0: only the pages the requests use).
    ragged=True makes prompt lengths not page-aligned. poison=True fills every slot that holds no token with NaN,
    so that reading an invisible slot shows up in the output. seed_offset selects an independent replica (a
    different layer of the same model).
    """
    device = torch.device(device)
    cfg_id = CONFIGS.index(name) + 1
    seed = SEED_BASE + cfg_id + 1000 * seed_offset
    g = _gen(device, seed)
    g_cpu = _gen("cpu", seed + 7)

    def L_of(full):
        L = max(64, int(round(full * scale)))
        if ragged:
            L = L - 5 if L % PAGE == 0 else L
        return L

    spans = span_offsets = None
    per_kv_head = True
    n_needles = 0
    if name == "tiny":
        dtype, R, Hq, Hkv, d, sigma = torch.float32, 1, 8, 2, 64, 1.0 / 8.0
        lens = [L_of(1024)]
        ark = [(1, 2, 5)]
        k_prop, n_q = 1, [4]
        n_needles = 2
        pool_min = 128
    elif name == "llama":
        dtype, R, Hq, Hkv, d, sigma = torch.bfloat16, 4, 32, 8, 128, 1.0
        lens = [L_of(32768)] * R
        N = (lens[0] + PAGE - 1) // PAGE
        k = max(1, int(round(0.0625 * N)) - 3) if scale < 1 else 125
        ark = [(1, 2, k)] * R
        k_prop, n_q = 4, [4] * R
        n_needles = 16
        pool_min = 0
    elif name == "long":
        dtype, R, Hq, Hkv, d, sigma = torch.bfloat16, 1, 40, 8, 128, 1.0
        lens = [L_of(131072)]
        ark = [(1, 4, 0)]
        k_prop, n_q = 8, [8]
        per_kv_head = False
        pool_min = 0
    elif name == "early":
        dtype, Hq, Hkv, d, sigma = torch.bfloat16, 32, 8, 128, 1.0
        R = batch if batch is not None else 1
        lens = [L_of(40960)] * R
        ark = [(0, 0, 8)] * R
        k_prop, n_q = 1, [1] * R
        n_needles = 4
        pool_min = 0
    elif name == "mixed":
        dtype, Hq, Hkv, d, sigma = torch.bfloat16, 32, 8, 128, 1.0
        R = batch if batch is not None else max(2, int(round(32 * min(1.0, scale * 4))))
        lo, hi = math.log(4096 * scale), math.log(131072 * scale)
        u = torch.rand(R, generator=g_cpu, dtype=torch.float64)
        lens = [max(64, int(math.floor(math.exp(lo + (hi - lo) * float(x))))) for x in u]
        if ragged:
            lens = [L - 5 if L % PAGE == 0 else L for L in lens]
        s_choices = [0.02, 0.055, 0.10, 0.25]
        splits = [(1, 2), (4, 4), (0, 0)]
        si = torch.randint(0, 4, (R,), generator=g_cpu).tolist()
        pi = torch.randint(0, 3, (R,), generator=g_cpu).tolist()
        ark = []
        for L, i, j in zip(lens, si, pi):
            N = (L + PAGE - 1) // PAGE
            a, r = splits[j]
            total = min(N, max(a + r + 1, int(math.floor(s_choices[i] * N + 0.5))))
            ark.append((a, r, max(0, total - a - r)))
        k_prop = 1
        n_q = [[2, 4, 8][t] for t in torch.randint(0, 3, (R,), generator=g_cpu).tolist()]
        n_needles = 5
        pool_min = 1 << 20 if scale >= 1 else 0
    else:
        raise ValueError(f"unknown workload {name!r}")
    if n_q_override is not None:
        n_q = [n_q_override] * R
    if pool_min_override is not None:
        pool_min = pool_min_override
    if k_prop_override is not None:
        k_prop = k_prop_override

    # Pages: prompt pages plus the tail pages the cycle writes (proposal tokens and the verify window).
    horizon = max(k_prop, max(n_q))
    pages_per_req = [(L + horizon + PAGE - 1) // PAGE for L in lens]
    max_pages = max(pages_per_req)
    need = sum(pages_per_req)
    P = max(pool_min, need + 64) if name != "tiny" else max(pool_min, need)
    perm = torch.randperm(P, generator=g_cpu)[:need].to(torch.int32)
    bt = torch.full((R, max_pages), -1, dtype=torch.int32)
    o = 0
    for r, npg in enumerate(pages_per_req):
        bt[r, :npg] = perm[o:o + npg]
        o += npg

    # Queries. The routing query is the first proposal query (or a noisy proxy of it for `early`).
    q_prop = _randn((k_prop, R, Hq, d), g, device, sigma)
    q_route = q_prop[0].clone()
    if name == "early":
        q_route = q_route + _randn((R, Hq, d), g, device, 0.3)

    # KV pool: every slot poisoned, then the prompt tokens of each request written.
    K = torch.empty((P, Hkv, PAGE, d), dtype=dtype, device=device)
    V = torch.empty((P, Hkv, PAGE, d), dtype=dtype, device=device)
    if poison:
        K.fill_(float("nan"))
        V.fill_(float("nan"))
    else:
        K.zero_()
        V.zero_()
    needles = []
    G = Hq // Hkv
    for r, L in enumerate(lens):
        N = (L + PAGE - 1) // PAGE
        kr = _randn((N, Hkv, PAGE, d), g, device, sigma)
        vr = _randn((N, Hkv, PAGE, d), g, device, sigma)
        nd = []
        if n_needles and N > 8:
            a, rr = ark[r][0], ark[r][1]
            lo_p, hi_p = max(a, 1), max(max(a, 1) + 1, N - max(rr, 1))
            cand = torch.randperm(hi_p - lo_p, generator=g_cpu)[: min(n_needles, hi_p - lo_p)] + lo_p
            nd = sorted(int(x) for x in cand)
            # Direction of each KV head's query group: the needle keys move 3 sigma along it.
            qg = q_route[r].view(Hkv, G, d).sum(dim=1)
            qhat = qg / qg.norm(dim=-1, keepdim=True).clamp_min(1e-30)
            for p in nd:
                kr[p] += 3.0 * sigma * qhat[:, None, :]
        needles.append(nd)
        kr = kr.to(dtype)
        vr = vr.to(dtype)
        tail = N * PAGE - L
        if tail and poison:
            kr[N - 1, :, PAGE - tail:, :] = float("nan")
            vr[N - 1, :, PAGE - tail:, :] = float("nan")
        idx = bt[r, :N].to(device=device, dtype=torch.int64)
        K.index_copy_(0, idx, kr)
        V.index_copy_(0, idx, vr)
        del kr, vr

    if name == "long":
        N = (lens[0] + PAGE - 1) // PAGE
        if scale >= 1:
            sp = _spans_long(g_cpu, N)
        else:
            n_spans = max(1, round(30 * N / 8192))
            total = max(8 * n_spans, round(446 * N / 8192))
            sp = _spans_long(g_cpu, N, n_spans=n_spans, total=total)
        spans = torch.tensor(sp, dtype=torch.int32)
        span_offsets = torch.tensor([0, len(sp)], dtype=torch.int32)

    k_new_prop = _randn((k_prop, R, Hkv, d), g, device, sigma).to(dtype)
    v_new_prop = _randn((k_prop, R, Hkv, d), g, device, sigma).to(dtype)
    q_offsets = torch.zeros(R + 1, dtype=torch.int32)
    q_offsets[1:] = torch.cumsum(torch.tensor(n_q, dtype=torch.int32), 0)
    tq = int(q_offsets[-1])
    q_ver = _randn((tq, Hq, d), g, device, sigma).to(dtype)
    k_new_ver = _randn((tq, Hkv, d), g, device, sigma).to(dtype)
    v_new_ver = _randn((tq, Hkv, d), g, device, sigma).to(dtype)

    # Decode-loop proxies of the early workload: the proxy of step t > 0 is its query plus fresh N(0, 0.3^2) noise,
    # drawn after everything above so that the other tensors do not depend on the number of steps.
    q_route_steps = None
    if name == "early":
        q_route_steps = torch.empty((k_prop, R, Hq, d), dtype=torch.float32, device=device)
        q_route_steps[0] = q_route
        if k_prop > 1:
            q_route_steps[1:] = q_prop[1:] + _randn((k_prop - 1, R, Hq, d), g, device, 0.3)
        q_route_steps = q_route_steps.to(dtype)

    dev = lambda t: t.to(device) if t is not None else None  # noqa: E731
    return Workload(
        name=name, dtype=dtype, R=R, Hq=Hq, Hkv=Hkv, d=d, num_pages=P, K=K, V=V,
        block_table=dev(bt), ctx_len=dev(torch.tensor(lens, dtype=torch.int32)),
        seq_len0=dev(torch.tensor(lens, dtype=torch.int32)), k_prop=k_prop,
        q_prop=q_prop.to(dtype), q_route=q_route.to(dtype), k_new_prop=k_new_prop, v_new_prop=v_new_prop,
        n_q=dev(torch.tensor(n_q, dtype=torch.int32)), q_offsets=dev(q_offsets), q_ver=q_ver,
        k_new_ver=k_new_ver, v_new_ver=v_new_ver, ark=dev(torch.tensor(ark, dtype=torch.int32)),
        per_kv_head=per_kv_head, spans=dev(spans), span_offsets=dev(span_offsets), needles=needles,
        sigma=sigma, q_route_steps=q_route_steps)


def make_prior(w: Workload, num_layers: int = 32, device="cpu", seed_offset: int = 0,
               needle_lift: float = 3.0, quantize: Optional[float] = None) -> torch.Tensor:
    """Seeded external-prior affinities for workload `w`: [R][num_layers][Hkv][max_pages] fp32.

    Stands in for a baked KRI prior (block_affinities[L][H][N] per request prefix): N(0, 1) per (layer, head,
    block), with every needle page of the request lifted by `needle_lift` in all layers and heads, so that a prior
    that "knows" the evidence favours those pages. Columns at or past a request's prompt pages are filled too; the
    selection ignores them. quantize = q rounds every value to a multiple of q, which makes pooled scores tie.
    """
    R, Hkv = w.R, w.Hkv
    max_pages = int(w.block_table.shape[1])
    g = _gen("cpu", SEED_BASE + 77 + 1000 * seed_offset)
    aff = torch.randn(R, num_layers, Hkv, max_pages, generator=g, dtype=torch.float32)
    for r, nd in enumerate(w.needles):
        if nd:
            aff[r, :, :, torch.tensor(nd, dtype=torch.long)] += needle_lift
    if quantize is not None:
        aff = torch.round(aff / quantize) * quantize
    return aff.to(device)


def make_verify_logits(w: Workload, vocab: int = 128256, accept: float = 0.95, device="cpu", seed_offset: int = 0,
                       dtype=torch.float32, ties: bool = False):
    """Seeded verifier logits for the windows of workload `w` (the carry row plus k = n_q - 1 proposals each).

    Returns (logits [total_rows][vocab], tokens [total_rows] int32, window offsets [R+1] int32). Token 0 of a window
    is the carry, drawn uniformly; each later token is a proposal. Background logits are N(0, 1). For each proposal
    the generator decides, with probability `accept`, that it should pass: its logit in the row before it is set to
    8 + U(0, 1) (far above the background), else to -8. ties=True draws the background from {0, 1, 2} instead, so
    that many tokens share a logit. Nothing here ranks tokens: the decision is planted in the data.
    """
    g = _gen("cpu", SEED_BASE + 91 + 1000 * seed_offset)
    n_q = w.n_q.cpu().tolist()
    offs = [0]
    for n in n_q:
        offs.append(offs[-1] + int(n))
    rows = offs[-1]
    if ties:
        lg = torch.randint(0, 3, (rows, vocab), generator=g).to(torch.float32)
    else:
        lg = torch.randn(rows, vocab, generator=g, dtype=torch.float32)
    tok = torch.randint(0, vocab, (rows,), generator=g, dtype=torch.int64)
    u = torch.rand(rows, generator=g, dtype=torch.float64)
    lift = torch.rand(rows, generator=g, dtype=torch.float32)
    for r in range(len(n_q)):
        for j in range(offs[r] + 1, offs[r + 1]):
            lg[j - 1, tok[j]] = (8.0 + float(lift[j])) if float(u[j]) < accept else -8.0
    return (lg.to(dtype).to(device), tok.to(torch.int32).to(device),
            torch.tensor(offs, dtype=torch.int32, device=device))
