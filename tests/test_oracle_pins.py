"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test ties an oracle function to something other than itself: the KRI page's worked A<a>R<r>K<k> example,
closed forms of softmax attention, torch's fp64 scaled_dot_product_attention on a dense gather, brute force on
tiny inputs, exact integer arithmetic, and the algebra of the KAP cost model.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGE = 16


# ----------------------------------------------------------------------------------------------- A/R/K top-K
def _read_ark_fixture():
    tags = {}
    for line in open(os.path.join(GOLDEN, "ark_128_block_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "num_blocks":
            n = int(f[1])
        elif f[0] == "budget":
            budget = int(f[1])
        elif f[0] == "tag":
            kv = dict(zip(f[2::2], f[3::2]))
            pinned = [] if kv["pinned"] == "-" else [int(x) for x in kv["pinned"].split(",")]
            tags[f[1]] = dict(a=int(kv["anchor"]), r=int(kv["recent"]), k=int(kv["k"]), pinned=pinned,
                              mid=(int(kv["middle_first"]), int(kv["middle_last"])))
    return n, budget, tags


@pytest.mark.parametrize("tag", ["A1R2K13", "A0R0K16", "A4R4K8"])
def test_ark_worked_example(orc, tag):
    n, budget, tags = _read_ark_fixture()
    t = tags[tag]
    assert t["a"] + t["r"] + t["k"] == budget
    rng = np.random.default_rng(5)
    scores = rng.standard_normal(n).astype(np.float32)
    sel = orc.topk_ark(scores, n, t["a"], t["r"], t["k"])
    assert len(sel) == budget
    assert list(sel) == sorted(sel)
    for p in t["pinned"]:
        assert p in sel
    lo, hi = t["mid"]
    chosen = [j for j in sel if j not in t["pinned"]]
    assert all(lo <= j <= hi for j in chosen)
    best = sorted(range(lo, hi + 1), key=lambda j: -float(scores[j]))[: t["k"]]
    assert sorted(best) == chosen


def test_ark_ties_go_to_lower_page(orc):
    scores = np.zeros(40, dtype=np.float32)
    scores[[7, 9, 30, 31]] = 2.0
    sel = orc.topk_ark(scores, 40, 1, 1, 3)
    assert list(sel) == [0, 7, 9, 30, 39]
    # all equal: the lowest middle ids win
    sel = orc.topk_ark(np.ones(20, np.float32), 20, 2, 3, 4)
    assert list(sel) == [0, 1, 2, 3, 4, 5, 17, 18, 19]


def test_ark_signed_zero_and_nan(orc):
    s = np.array([0, -0.0, 0.0, np.nan, -1.0, 0.0], dtype=np.float32)
    # -0 and +0 tie (the lower id wins); NaN ranks below -1
    assert list(orc.topk_ark(s, 6, 0, 0, 2)) == [0, 1]
    assert list(orc.topk_ark(s, 6, 0, 0, 5)) == [0, 1, 2, 4, 5]


def test_ark_small_and_degenerate(orc):
    s = np.arange(10, dtype=np.float32)
    assert list(orc.topk_ark(s, 3, 1, 2, 5)) == [0, 1, 2]          # N <= a + r: everything pinned
    assert list(orc.topk_ark(s, 10, 2, 2, 0)) == [0, 1, 8, 9]      # k = 0: the anchor+recency hybrid
    assert list(orc.topk_ark(s, 10, 0, 3, 0)) == [7, 8, 9]         # recency only
    assert list(orc.topk_ark(s, 10, 0, 0, 100)) == list(range(10))  # k beyond the middle keeps everything
    assert list(orc.topk_ark(s, 1, 0, 0, 1)) == [0]


def test_ark_random_brute_force(orc):
    rng = np.random.default_rng(11)
    for _ in range(200):
        n = int(rng.integers(1, 90))
        a, r, k = (int(x) for x in rng.integers(0, 6, 3))
        s = rng.integers(-3, 4, n).astype(np.float32)  # many ties
        sel = orc.topk_ark(s, n, a, r, k)
        pinned = set(range(min(a, n))) | set(range(max(0, n - r), n))
        mid = [j for j in range(n) if j not in pinned]
        mid.sort(key=lambda j: (-float(s[j]), j))
        assert list(sel) == sorted(pinned | set(mid[:k]))


# --------------------------------------------------------------------------------------------- summaries
def test_summary_is_block_mean(orc):
    rng = np.random.default_rng(0)
    P, hkv, d = 12, 2, 64
    K = rng.integers(-8, 9, (P, hkv, PAGE, d)).astype(np.float32)   # integer values: sums are exact
    bt = np.array([[3, 7, 1, 0], [5, 2, 9, -1]], np.int32)
    ctx = np.array([64, 37], np.int32)                                  # second request: partial last page
    K[9, :, 37 - 32:, :] = np.nan                                         # invalid slots of that page
    S = orc.build_summaries(K, bt, ctx)
    for r in range(2):
        for j in range((ctx[r] + 15) // 16):
            n = min(16, ctx[r] - 16 * j)
            want = K[bt[r, j], :, :n, :].astype(np.float64).mean(axis=1)
            got = S[bt[r, j]].astype(np.float64)
            if n == 16:
                assert np.array_equal(got, want)  # division by 16 is exact
            else:
                np.testing.assert_allclose(got, want, rtol=2 ** -23, atol=0)
            assert np.isfinite(got).all()


# ----------------------------------------------------------------------------------------------- scores
def test_dot_fixed_order_exact_on_integers(orc):
    rng = np.random.default_rng(1)
    for d in (64, 128):
        a = rng.integers(-50, 51, d).astype(np.float32)
        b = rng.integers(-50, 51, d).astype(np.float32)
        assert float(orc.dot_fixed_order(a, b)) == float(np.dot(a.astype(np.int64), b.astype(np.int64)))


def test_dot_fixed_order_is_the_stated_order(orc):
    # 2^24 + 1 rounds back to 2^24 inside partial 0 (i = 0 and i = 32), and partial 16 holds -2^24: the stated order
    # gives 0 where an exact or sequential sum gives 1. A different lane assignment or combine order fails here.
    a = np.zeros(64, np.float32)
    b = np.ones(64, np.float32)
    a[0], a[32], a[16] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    assert float(orc.dot_fixed_order(a, b)) == 0.0
    a2 = a.copy()
    a2[32], a2[48] = 0.0, 1.0   # the 1 now sits in partial 16 next to -2^24: -2^24 + 1 is exact, result 1
    assert float(orc.dot_fixed_order(a2, b)) == 1.0


def test_scores_exact_on_integers(orc):
    rng = np.random.default_rng(2)
    R, hq, hkv, d, P = 2, 8, 2, 64, 10
    q = rng.integers(-4, 5, (R, hq, d)).astype(np.float32)
    S = rng.integers(-4, 5, (P, hkv, d)).astype(np.float32)
    bt = np.array([[4, 1, 7], [0, 9, 2]], np.int32)
    ctx = np.array([48, 40], np.int32)
    G = hq // hkv
    per, per64 = orc.scores(q, S, bt, ctx, per_head=True)
    pooled, _ = orc.scores(q, S, bt, ctx, per_head=False)
    for r in range(R):
        for j in range(3):
            tot = 0
            for h in range(hkv):
                qbar = q[r, h * G:(h + 1) * G].astype(np.int64).sum(axis=0)
                v = int(np.dot(qbar, S[bt[r, j], h].astype(np.int64)))
                assert per[r, h, j] == v and per64[r, h, j] == v
                tot += v
            assert pooled[r, 0, j] == tot


def test_scores_fp32_close_to_fp64(orc):
    rng = np.random.default_rng(3)
    R, hq, hkv, d, P = 1, 32, 8, 128, 40
    q = rng.standard_normal((R, hq, d)).astype(np.float32)
    S = rng.standard_normal((P, hkv, d)).astype(np.float32)
    bt = rng.permutation(P)[:32].astype(np.int32)[None]
    ctx = np.array([512], np.int32)
    s32, s64 = orc.scores(q, S, bt, ctx, per_head=True)
    assert np.abs(s32[:, :, :32] - s64[:, :, :32]).max() < 1e-4 * np.abs(s64[:, :, :32]).max()


# ------------------------------------------------------------------------------------------------ spans
# ------------------------------------------------------------------ external-prior scores (KRI prior schema)
def test_prior_scores_exact_mean_on_dyadic_values(orc):
    """Integer affinities with L*H a power of two: every partial sum and the division are exact, so the pooled score
    is the exact arithmetic mean over layers and heads (KRI page: the connector mean-pools block_affinities)."""
    rng = np.random.default_rng(11)
    for L, H in [(1, 1), (4, 8), (8, 8), (32, 8), (2, 16)]:
        aff = rng.integers(-1000, 1000, size=(L, H, 37)).astype(np.float32)
        got = orc.prior_scores(aff)
        want = aff.astype(np.float64).sum(axis=(0, 1)) / (L * H)
        assert np.array_equal(got.astype(np.float64), want), (L, H)


def test_prior_scores_chunked_order_hand_value(orc):
    """The stated order sums 32 rows at a time: one huge value and 31 ones in the first chunk lose the ones, the
    second chunk's 32 ones survive as 32. Worked by hand: (2^25 + 32) / 64 = 524288.5. A plain running sum would lose
    all 63 ones (524288.0), a pairwise or fp64 sum would keep them (524288.984...)."""
    aff = np.ones((8, 8, 1), dtype=np.float32)
    aff[0, 0, 0] = 2.0 ** 25
    assert orc.prior_scores(aff)[0] == np.float32(524288.5)
    # Row index i = l*H + h: the huge value at (l=3, h=7) is row 31, the last of chunk 0, where the 31 ones before it
    # round up to 32 (spacing 4 at 2^25); chunk 1 adds 32: (2^25 + 64) / 64 = 524289. With rows taken as h*L + l it
    # would be row 59 and give 524288.9375.
    aff = np.ones((8, 8, 1), dtype=np.float32)
    aff[3, 7, 0] = 2.0 ** 25
    assert orc.prior_scores(aff)[0] == np.float32(524289.0)


def test_prior_scores_within_fp32_summation_bound(orc):
    """Random affinities: the fp32 pooled score is within the recursive-summation bound of the exact mean."""
    rng = np.random.default_rng(12)
    L, H, N = 32, 8, 257
    aff = rng.standard_normal((L, H, N)).astype(np.float32)
    got = orc.prior_scores(aff).astype(np.float64)
    a64 = aff.astype(np.float64)
    exact = a64.sum(axis=(0, 1)) / (L * H)
    bound = (L * H + 2) * 2.0 ** -24 * np.abs(a64).sum(axis=(0, 1)) / (L * H) + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(got - exact) <= bound)


def test_prior_selection_keeps_planted_blocks(orc):
    """A/R/K over pooled priors: blocks whose affinity is raised in every layer and head are the k chosen, next to
    the pinned anchor and recent blocks (KRI page, A1R2K13 over a 128-block prefix)."""
    rng = np.random.default_rng(13)
    L, H, N = 4, 8, 128
    aff = rng.standard_normal((L, H, N)).astype(np.float32)
    planted = np.sort(rng.choice(np.arange(1, 126), size=13, replace=False))
    aff[:, :, planted] += 20.0
    ids = orc.topk_ark(orc.prior_scores(aff), N, 1, 2, 13)
    assert list(ids) == sorted([0] + planted.tolist() + [126, 127])


# ------------------------------------------------------- tolerant acceptance and commit (KAP paper, verifier)
def test_accept_commit_worked_windows(orc):
    """Hand-worked windows of a 5-token vocabulary (carry, then proposals; row j predicts after token j)."""
    lg = np.array([[0, 5, 4, 3, 1], [9, 8, 7, 6, 5], [1, 1, 1, 1, 1]], np.float32)
    # token 3 is third in row 0 (5, 4, 3): accepted; token 2 is third in row 1: accepted; all-equal row 2 -> token 0
    assert orc.accept_commit(lg, [0, 3, 2], 3, 100) == (2, 0, 103)
    # token 4 is fourth in row 0: rejected at once; the carry is row 0's first (token 1); only the carry commits
    assert orc.accept_commit(lg, [0, 4, 2], 3, 100) == (0, 1, 101)
    # the second proposal fails (token 0 is fifth in row 1) after the first passes: carry = first of row 1 (token 0)
    assert orc.accept_commit(lg, [0, 1, 4], 3, 7) == (1, 0, 9)
    # a token outside the vocabulary is rejected
    assert orc.accept_commit(lg, [0, 5, 2], 3, 0) == (0, 1, 1)


def test_accept_commit_greedy_special_case(orc):
    """With n = 1 the rule is greedy speculative verification: the accepted prefix is the longest run where each
    proposal equals the argmax of the row before it, and the carry is the argmax after that prefix."""
    rng = np.random.default_rng(21)
    for _ in range(300):
        rows, V = int(rng.integers(1, 7)), int(rng.integers(1, 9))
        lg = rng.integers(0, 4, size=(rows, V)).astype(np.float32)
        am = lg.argmax(axis=1)   # first maximum: lower id on ties
        toks = [0] + [int(am[j - 1]) if rng.random() < 0.7 else int(rng.integers(0, V)) for j in range(1, rows)]
        m = 0
        while m + 1 < rows and toks[m + 1] == am[m]:
            m += 1
        assert orc.accept_commit(lg, toks, 1, 50) == (m, int(am[m]), 51 + m)


def test_accept_commit_counting_brute_force(orc):
    """Random tied and NaN logits: a proposal passes iff fewer than n tokens beat it (a higher logit, or an equal one
    with a lower id; NaN beats nothing and loses to every number)."""
    rng = np.random.default_rng(22)

    def beats(a, ia, b, ib):  # does (a, ia) come before (b, ib)?
        if np.isnan(a):
            return bool(np.isnan(b)) and ia < ib
        if np.isnan(b):
            return True
        return a > b or (a == b and ia < ib)

    for _ in range(300):
        rows, V, n = int(rng.integers(2, 6)), int(rng.integers(2, 10)), int(rng.integers(1, 5))
        lg = rng.integers(0, 3, size=(rows, V)).astype(np.float32)
        lg[rng.random((rows, V)) < 0.15] = np.nan
        toks = [int(rng.integers(0, V)) for _ in range(rows)]
        m = 0
        for j in range(1, rows):
            x = toks[j]
            nb = sum(beats(lg[j - 1, t], t, lg[j - 1, x], x) for t in range(V) if t != x)
            if nb >= n:
                break
            m += 1
        first = [t for t in range(V) if not any(beats(lg[m, u], u, lg[m, t], t) for u in range(V) if u != t)]
        assert orc.accept_commit(lg, toks, n, 3) == (m, first[0], 4 + m)


def test_accept_commit_everything_passes_with_n_at_least_v(orc):
    rng = np.random.default_rng(23)
    lg = rng.standard_normal((5, 6)).astype(np.float32)
    m, c, sl = orc.accept_commit(lg, [1, 2, 3, 4, 5], 6, 10)
    assert (m, sl) == (4, 15) and c == int(lg[4].argmax())


# -------------------------------------------------- materialised compact workspace (KAP paper, compiler / fallback)
def test_materialize_row_layout_and_fallback(orc):
    """Selected entries go to consecutive workspace pages from the request's base, in access order; tail entries keep
    their pages; a selected page that also holds positions at or past ctx_len stays in place (generated tokens are
    written into it through the full table later); a selection larger than the workspace is left as it is."""
    row, lp = [5, 9, 2, 40, 41], [0, 3, 6, 7, 8]
    out, pairs, fits = orc.materialize_row(row, lp, 5, 3, 112, 100, 8)     # 112 = 7 full pages: 0, 3, 6 all prompt
    assert fits and out.tolist() == [100, 101, 102, 40, 41] and pairs == [(5, 100), (9, 101), (2, 102)]
    out, pairs, fits = orc.materialize_row(row, lp, 5, 3, 100, 100, 8)     # page 6 holds positions 96..111 > 100
    assert fits and out.tolist() == [100, 101, 2, 40, 41] and pairs == [(5, 100), (9, 101)]
    out, pairs, fits = orc.materialize_row(row, lp, 5, 3, 112, 100, 2)
    assert not fits and out.tolist() == row and pairs == []
    out, pairs, fits = orc.materialize_row(row, lp, 5, 0, 112, 100, 2)
    assert fits and out.tolist() == row and pairs == []


def test_materialized_view_keeps_attention_exact(orc):
    """Copying the selected pages into the workspace and pointing the table there leaves proposal attention
    unchanged bit for bit: the same values sit at the same logical positions (one view shared by all heads)."""
    R, hq, hkv, d = 2, 8, 2, 64
    ctx = np.array([70, 100], np.int32)
    seq = ctx + 3
    rng, bt, K, V = _toy(30, R, hq, hkv, d, tuple(ctx))
    P0 = K.shape[0]
    ws_pages = 6
    K2 = np.concatenate([K, np.full((R * ws_pages,) + K.shape[1:], np.nan, np.float32)])
    V2 = np.concatenate([V, np.full((R * ws_pages,) + V.shape[1:], np.nan, np.float32)])
    q = rng.standard_normal((R, hq, d)).astype(np.float32)
    cap = 5
    sel = np.zeros((R, 1, cap), np.int32)
    nsel = np.zeros((R, 1), np.int32)
    bt2 = bt.copy()
    for r in range(R):
        N = (ctx[r] + 15) // 16
        s = sorted(rng.choice(N, size=4, replace=False).tolist())
        sel[r, 0, :4] = s
        nsel[r, 0] = 4
        out_row, pairs, fits = orc.materialize_row(bt[r, s], s, 4, 4, int(ctx[r]), P0 + r * ws_pages, ws_pages)
        assert fits
        for src, dst in pairs:
            K2[dst], V2[dst] = K[src], V[src]
        for i, lp in enumerate(s):
            bt2[r, lp] = out_row[i]
    o1, l1 = orc.attn_propose(q, K, V, bt, ctx, seq, sel, nsel)
    o2, l2 = orc.attn_propose(q, K2, V2, bt2, ctx, seq, sel, nsel)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_select_spans_brute_force(orc):
    rng = np.random.default_rng(4)
    for _ in range(100):
        N = int(rng.integers(1, 60))
        ns = int(rng.integers(0, 5))
        spans = [(int(rng.integers(0, N * 16 + 20)), int(rng.integers(0, 40))) for _ in range(ns)]
        a, r = (int(x) for x in rng.integers(0, 3, 2))
        want = set(range(min(a, N))) | set(range(max(0, N - r), N))
        for first, ln in spans:
            for t in range(first, first + ln):
                if t < N * 16:
                    want.add(t // 16)
        got = orc.select_spans(N, np.array(spans, np.int32).reshape(-1, 2), a, r)
        assert list(got) == sorted(want)


# ------------------------------------------------------------------------------------- view and slots
def test_compile_view_invariants(orc):
    rng = np.random.default_rng(6)
    for _ in range(100):
        ctx = int(rng.integers(1, 400))
        horizon = int(rng.integers(0, 20))
        seq = ctx + int(rng.integers(0, 10))
        npages = (seq + horizon + 15) // 16 + 1
        bt = rng.permutation(1000)[:npages].astype(np.int32)
        N = (ctx + 15) // 16
        sel = sorted(set(int(x) for x in rng.integers(0, N, int(rng.integers(1, N + 1)))))
        cbt, clog, nsel = orc.compile_view_row(bt, ctx, seq, horizon, np.array(sel, np.int32))
        assert nsel == len(sel)
        assert list(clog[:nsel]) == sel
        assert np.all(np.diff(clog) > 0)                       # access order == logical order, no duplicates
        assert np.array_equal(cbt, bt[clog])                    # logical positions preserved
        tail = [j for j in range(ctx // 16, npages) if j * 16 < seq + horizon]
        assert sorted(set(clog)) == sorted(set(sel) | set(tail))
        # KRI connector skip list: the selected prompt blocks and their sorted complement partition range(N)
        skip = sorted(b for b in range(N) if b not in set(sel))
        assert sorted(set(sel) | set(skip)) == list(range(N)) and not (set(sel) & set(skip))


def test_slot_mapping_inverts_through_the_table(orc):
    rng = np.random.default_rng(7)
    bt = rng.permutation(300)[:20].astype(np.int32)
    inverse = {int(p): j for j, p in enumerate(bt)}
    for pos in range(0, 20 * 16):
        s = orc.slot(bt, pos)
        page, off = divmod(s, 16)
        assert inverse[page] * 16 + off == pos
    assert orc.slot(bt, 20 * 16) == -1
    bt2 = bt.copy()
    bt2[3] = -1
    assert orc.slot(bt2, 3 * 16 + 5) == -1


# ------------------------------------------------------------------------------------------------- RoPE
def test_inv_freq_closed_form(orc):
    for d in (64, 128):
        f = orc.inv_freq(d, 1.0e4).astype(np.float64)
        assert f[0] == 1.0
        assert abs(f[d // 4] - 0.01) <= 0.01 * 2 ** -23        # theta^(-1/2) = 0.01
        ratio = f[1:] / f[:-1]
        np.testing.assert_allclose(ratio, 1.0e4 ** (-2.0 / d), rtol=3e-7)


def test_rope_properties(orc):
    rng = np.random.default_rng(8)
    d = 64
    f = orc.inv_freq(d)
    x = rng.standard_normal((5, 3, d)).astype(np.float32)
    y0 = orc.rope(x, np.zeros(5, np.int32), f)
    np.testing.assert_array_equal(y0, x.astype(np.float64))      # position 0 is the identity
    pos = np.array([1, 17, 1000, 65535, 131071], np.int32)
    y = orc.rope(x, pos, f)
    h = d // 2
    np.testing.assert_allclose(y[..., :h] ** 2 + y[..., h:] ** 2,
                               x[..., :h].astype(np.float64) ** 2 + x[..., h:].astype(np.float64) ** 2,
                               rtol=1e-12, atol=1e-12)            # each pair keeps its norm
    # complex-number form: (x_i + i x_{i+d/2}) * exp(i * angle), angle formed in fp32
    ang = (pos.astype(np.float32)[:, None] * f[None, :]).astype(np.float64)
    z = (x[..., :h].astype(np.float64) + 1j * x[..., h:].astype(np.float64)) * np.exp(1j * ang)[:, None, :]
    np.testing.assert_allclose(y[..., :h], z.real, atol=1e-12)
    np.testing.assert_allclose(y[..., h:], z.imag, atol=1e-12)


def test_rope_relative_position(orc):
    rng = np.random.default_rng(9)
    d = 128
    f = orc.inv_freq(d)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, d)).astype(np.float32)
    def dot(m, n):
        return float(np.sum(orc.rope(q, np.array([m], np.int32), f) * orc.rope(k, np.array([n], np.int32), f)))
    base = dot(10, 3)
    for c in (1, 5, 100, 2000):
        assert abs(dot(10 + c, 3 + c) - base) < 1e-3 * (1 + abs(base))


# -------------------------------------------------------------------------------------------- attention
def _dense(K, bt_row, n_tok, h):
    """Gathers positions 0..n_tok-1 of KV head h through one block-table row into a dense [n_tok][d] array."""
    return np.stack([K[bt_row[p // 16], h, p % 16] for p in range(n_tok)]).astype(np.float64)


def _sdpa(q, k, v, mask):
    """torch fp64 scaled_dot_product_attention plus its log-sum-exp (the library routine the oracle must match)."""
    qt = torch.from_numpy(q)[None, None, None]   # [1,1,1,d]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = torch.from_numpy(mask)[None, None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m)[0, 0, 0].numpy()
    logits = (k @ q) / math.sqrt(q.shape[0])
    lse = float(torch.logsumexp(torch.from_numpy(logits[mask]), 0))
    return o, lse


def _toy(seed, R=2, hq=8, hkv=2, d=64, ctx=(70, 100), extra=4, poison=True):
    rng = np.random.default_rng(seed)
    npg = [(c + extra + 15) // 16 for c in ctx]
    P = sum(npg) + 3
    perm = rng.permutation(P)
    bt = np.full((R, max(npg)), -1, np.int32)
    o = 0
    for r in range(R):
        bt[r, :npg[r]] = perm[o:o + npg[r]]
        o += npg[r]
    K = rng.standard_normal((P, hkv, 16, d)).astype(np.float32)
    V = rng.standard_normal((P, hkv, 16, d)).astype(np.float32)
    return rng, bt, K, V


def test_propose_matches_sdpa_on_masked_subset(orc):
    R, hq, hkv, d = 2, 8, 2, 64
    ctx = np.array([70, 100], np.int32)
    seq = ctx + 3
    rng, bt, K, V = _toy(10, R, hq, hkv, d, tuple(ctx))
    # poison every slot at or past seq_len: the oracle must never read them
    for r in range(R):
        for p in range(seq[r], bt.shape[1] * 16):
            if bt[r, p // 16] >= 0:
                K[bt[r, p // 16], :, p % 16] = np.nan
                V[bt[r, p // 16], :, p % 16] = np.nan
    q = rng.standard_normal((R, hq, d)).astype(np.float32)
    cap = 7
    sel = np.zeros((R, hkv, cap), np.int32)
    nsel = np.zeros((R, hkv), np.int32)
    for r in range(R):
        N = (ctx[r] + 15) // 16
        for h in range(hkv):
            s = sorted(rng.choice(N, size=min(3 + h, N), replace=False))
            sel[r, h, :len(s)] = s
            nsel[r, h] = len(s)
    out, lse = orc.attn_propose(q, K, V, bt, ctx, seq, sel, nsel)
    G = hq // hkv
    for r in range(R):
        for h in range(hkv):
            n_tok = int(seq[r])
            k = _dense(K, bt[r], n_tok, h)
            v = _dense(V, bt[r], n_tok, h)
            chosen = set(sel[r, h, :nsel[r, h]].tolist())
            mask = np.array([(p >= ctx[r]) or (p // 16 in chosen) for p in range(n_tok)])
            for g in range(G):
                o, l = _sdpa(q[r, h * G + g].astype(np.float64), k, v, mask)
                np.testing.assert_allclose(out[r, h * G + g], o, atol=1e-12)
                assert abs(lse[r, h * G + g] - l) < 1e-12
    assert np.isfinite(out).all()


def test_propose_all_pages_equals_full_attention(orc):
    R, hq, hkv, d = 2, 8, 2, 64
    ctx = np.array([70, 100], np.int32)
    seq = ctx + 2
    rng, bt, K, V = _toy(12, R, hq, hkv, d, tuple(ctx))
    q = rng.standard_normal((R, hq, d)).astype(np.float32)
    cap = 8
    sel = np.zeros((R, 1, cap), np.int32)
    nsel = np.zeros((R, 1), np.int32)
    for r in range(R):
        N = (ctx[r] + 15) // 16
        sel[r, 0, :N] = np.arange(N)
        nsel[r, 0] = N
    out, lse = orc.attn_propose(q, K, V, bt, ctx, seq, sel, nsel)
    G = hq // hkv
    for r in range(R):
        for h in range(hkv):
            k = _dense(K, bt[r], int(seq[r]), h)
            v = _dense(V, bt[r], int(seq[r]), h)
            for g in range(G):
                o, l = _sdpa(q[r, h * G + g].astype(np.float64), k, v, np.ones(int(seq[r]), bool))
                np.testing.assert_allclose(out[r, h * G + g], o, atol=1e-12)
                assert abs(lse[r, h * G + g] - l) < 1e-12


def test_attention_closed_forms(orc):
    d, hkv, hq = 64, 1, 2
    rng = np.random.default_rng(13)
    K = rng.standard_normal((4, hkv, 16, d)).astype(np.float32)
    V = rng.standard_normal((4, hkv, 16, d)).astype(np.float32)
    q = rng.standard_normal((1, hq, d)).astype(np.float32)
    bt = np.array([[2, 0, 3]], np.int32)
    # one visible token: out = v, lse = its logit
    out, lse = orc.attn_verify(q, K, V, bt, np.array([0, 1], np.int32), np.array([0], np.int32))
    kk = K[2, 0, 0].astype(np.float64)
    for g in range(hq):
        np.testing.assert_allclose(out[0, g], V[2, 0, 0], atol=1e-12)
        assert abs(lse[0, g] - float(q[0, g].astype(np.float64) @ kk) / 8.0) < 1e-12
    # identical keys: uniform weights, out = mean of v, lse = logit + log(n)
    K2 = K.copy()
    K2[:, 0, :, :] = K[0, 0, 0]
    n = 37
    out, lse = orc.attn_verify(q, K2, V, bt, np.array([0, 1], np.int32), np.array([n - 1], np.int32))
    vs = _dense(V, bt[0], n, 0)
    for g in range(hq):
        np.testing.assert_allclose(out[0, g], vs.mean(axis=0), atol=1e-12)
        logit = float(q[0, g].astype(np.float64) @ K[0, 0, 0].astype(np.float64)) / 8.0
        assert abs(lse[0, g] - (logit + math.log(n))) < 1e-12


def test_verify_is_causal_and_matches_sdpa(orc):
    R, hq, hkv, d = 2, 8, 2, 64
    ctx = (70, 100)
    rng, bt, K, V = _toy(14, R, hq, hkv, d, ctx, extra=8)
    nq = [3, 5]
    qo = np.array([0, 3, 8], np.int32)
    qs = np.array([ctx[0], ctx[1] - 2], np.int32)
    q = rng.standard_normal((8, hq, d)).astype(np.float32)
    out, lse = orc.attn_verify(q, K, V, bt, qo, qs)
    G = hq // hkv
    for r in range(R):
        last = qs[r] + nq[r] - 1
        for h in range(hkv):
            k = _dense(K, bt[r], last + 1, h)
            v = _dense(V, bt[r], last + 1, h)
            for i in range(nq[r]):
                mask = np.arange(last + 1) <= qs[r] + i
                for g in range(G):
                    o, l = _sdpa(q[qo[r] + i, h * G + g].astype(np.float64), k, v, mask)
                    np.testing.assert_allclose(out[qo[r] + i, h * G + g], o, atol=1e-12)
                    assert abs(lse[qo[r] + i, h * G + g] - l) < 1e-12
    # changing the KV of a later candidate leaves earlier rows unchanged
    K3, V3 = K.copy(), V.copy()
    p = qs[1] + 3
    K3[bt[1, p // 16], :, p % 16] += 5.0
    V3[bt[1, p // 16], :, p % 16] -= 5.0
    out3, lse3 = orc.attn_verify(q, K3, V3, bt, qo, qs)
    np.testing.assert_array_equal(out3[:3 + 3], out[:3 + 3])
    assert not np.allclose(out3[3 + 3], out[3 + 3])


def test_verify_row_equals_decode_with_every_page(orc):
    R, hq, hkv, d = 1, 8, 2, 64
    rng, bt, K, V = _toy(15, 1, hq, hkv, d, (90,), extra=6)
    q = rng.standard_normal((4, hq, d)).astype(np.float32)
    out, lse = orc.attn_verify(q, K, V, bt, np.array([0, 4], np.int32), np.array([90], np.int32))
    for i in range(4):
        N = (90 + 15) // 16
        sel = np.arange(N, dtype=np.int32).reshape(1, 1, N)
        o2, l2 = orc.attn_propose(q[i:i + 1], K, V, bt, np.array([90], np.int32), np.array([91 + i], np.int32), sel,
                                  np.array([[N]], np.int32))
        np.testing.assert_allclose(out[i], o2[0], atol=1e-13)
        np.testing.assert_allclose(lse[i], l2[0], atol=1e-13)


# ------------------------------------------------------------------------------------------- cost model
def test_cost_model_boundary_algebra():
    from oracle import cost_model as cm
    rng = np.random.default_rng(16)
    for _ in range(2000):
        k = int(rng.integers(1, 12))
        h, s = float(rng.uniform(0, 1)), float(rng.uniform(0.001, 1))
        w, kv = float(rng.uniform(0.1, 10)), float(rng.uniform(0.1, 10))
        diff = cm.cost_base(k, h, w, kv) - cm.cost_plan(k, s, w, w, kv)
        assert abs(diff - k * ((h - s) * kv - (1 - h) * w)) < 1e-9 * (1 + abs(diff))
        if abs(diff) > 1e-9:
            assert (diff > 0) == cm.plan_wins(h, s, w, kv)
    # at KV_crit the two costs meet
    h, s, w = 0.95, 0.055, 3.0
    kvc = cm.kv_crit(h, s, w)
    assert abs(cm.cost_base(6, h, w, kvc) - cm.cost_plan(6, s, w, w, kvc)) < 1e-9
    assert cm.kv_crit(0.3, 0.4, 1.0) == float("inf")     # h <= s: no context length pays off


def test_cost_model_against_printed_points():
    from oracle import cost_model as cm
    pts = {}
    for line in open(os.path.join(GOLDEN, "kap_cost_points.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        pts[f[0]] = [float(x) for x in f[1:]]
    lo, hi = pts["h_range"]
    k = int(pts["k"][0])
    for ctx in ("4K", "128K"):
        s, margin, speedup = pts[ctx]
        h = s + margin
        assert lo - 0.01 <= h <= hi + 0.01             # printed s and h - s give the stated acceptance range
        assert h > s                                     # the necessary condition of the boundary
        # a measured speedup > 1 means the plan sits on the winning side: W_main / KV below (h - s) / (1 - h)
        assert speedup > 1.0
        w_over_kv_max = margin / (1.0 - h)
        assert cm.plan_wins(h, s, 0.99 * w_over_kv_max, 1.0)
        assert not cm.plan_wins(h, s, 1.01 * w_over_kv_max, 1.0)
    # the cycle's KV traffic at 128K retention: k proposals of s*KV plus one full read
    assert abs(cm.cycle_kv_bytes(k, 0.055, 1.0) - (1 + 6 * 0.055)) < 1e-12
