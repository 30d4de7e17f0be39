"""The benchmark's algorithmic byte model (bench.step_bytes) against the KAP paper's cost model, on CPU.

The cost model of a cycle with the weight terms set to zero is k*s*KV + KV (k proposals over the retained fraction s,
then one full verification). The byte model enumerates the selected pages instead; the two must agree up to the
tokens the cycle itself generates, which the cost model (fixed KV) leaves out. At the benchmark's shape the proposal
bytes must also lie within 2% of s*KV. Only metadata is built: no KV data is needed.
"""
import os
import sys
from types import SimpleNamespace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _layer(L, R=4, hkv=8, d=128, k_prop=4, n_q=4, a=1, r=2, k=125, seed=3):
    """Metadata of one benchmark layer: prompt lengths, window sizes and an A/R/K selection per (request, KV head)."""
    rng = np.random.default_rng(seed)
    N = (L + 15) // 16
    sel = np.zeros((R, hkv, a + r + k), np.int32)
    for rr in range(R):
        for h in range(hkv):
            mid = np.sort(rng.choice(np.arange(a, N - r), size=k, replace=False))
            sel[rr, h] = np.concatenate([np.arange(a), mid, np.arange(N - r, N)])
    w = SimpleNamespace(d=d, Hkv=hkv, R=R, k_prop=k_prop, ctx_len=torch.full((R,), L, dtype=torch.int32),
                        seq_len0=torch.full((R,), L, dtype=torch.int32), n_q=torch.full((R,), n_q, dtype=torch.int32))
    n_sel = torch.full((R, hkv), a + r + k, dtype=torch.int32)
    return w, torch.from_numpy(sel), n_sel


def test_byte_model_matches_the_cost_model():
    import bench
    from oracle import cost_model as cm
    for L in (32768, 32768 - 5):   # page-aligned prompt, and a partial last page (always kept: it is a recent page)
        w, sel, n_sel = _layer(L)
        b = bench.step_bytes(w, None, sel, n_sel)
        kv_tok = w.d * 2 * 2 * w.Hkv                  # K and V bytes of one position over all KV heads (bf16)
        KV = w.R * L * kv_tok                          # the full prompt KV the verifier reads
        full_pages = sel.shape[2] - 1                  # every selected page is full except the last prompt page
        last_valid = L - 16 * (((L + 15) // 16) - 1)
        s = (16 * full_pages + last_valid) / L         # retained fraction of prompt tokens
        generated = sum(w.R * (i + 1) * kv_tok for i in range(w.k_prop)) + w.R * 4 * kv_tok
        model = cm.cycle_kv_bytes(w.k_prop, s, KV)
        assert abs(sum(b["propose"]) + b["verify"] - (model + generated)) < 1e-6 * model


def test_proposal_bytes_within_two_percent_of_s_kv():
    import bench
    w, sel, n_sel = _layer(32768)
    b = bench.step_bytes(w, None, sel, n_sel)
    KV = w.R * 32768 * w.d * 2 * 2 * w.Hkv
    s = 128 / 2048
    for p in b["propose"]:
        assert abs(p - s * KV) <= 0.02 * s * KV
    assert b["score"] == w.R * 2048 * w.Hkv * w.d * 4   # one fp32 summary per (prompt page, KV head)


def test_byte_model_shared_view_long_context():
    """The long-context shape: one request, one view row shared by the 8 KV heads (rows_per_seq = 1). Every head
    reads the shared selection, so a proposal step reads Hkv x (selected prompt tokens + generated tokens) and the
    cycle matches the cost model with s = selected prompt tokens / L; each step is within 2% of s*KV."""
    import bench
    from oracle import cost_model as cm
    L, hkv, d, k_prop, n_q = 131072, 8, 128, 8, 8
    N = L // 16
    rng = np.random.default_rng(5)
    mid = np.sort(rng.choice(np.arange(1, N - 4), size=446, replace=False))
    pages = np.concatenate([[0], mid, np.arange(N - 4, N)]).astype(np.int32)   # 451 pages, s = 5.5%
    w = SimpleNamespace(d=d, Hkv=hkv, R=1, k_prop=k_prop, ctx_len=torch.tensor([L], dtype=torch.int32),
                        seq_len0=torch.tensor([L], dtype=torch.int32), n_q=torch.tensor([n_q], dtype=torch.int32))
    sel = torch.from_numpy(pages.reshape(1, 1, -1))
    n_sel = torch.tensor([[pages.size]], dtype=torch.int32)
    b = bench.step_bytes(w, None, sel, n_sel)
    kv_tok = d * 2 * 2 * hkv
    KV = L * kv_tok
    s = 16 * pages.size / L
    generated = sum((i + 1) * kv_tok for i in range(k_prop)) + n_q * kv_tok
    model = cm.cycle_kv_bytes(k_prop, s, KV)
    assert abs(sum(b["propose"]) + b["verify"] - (model + generated)) < 1e-6 * model
    for p in b["propose"]:
        assert abs(p - s * KV) <= 0.02 * s * KV
    assert b["score"] == N * hkv * d * 4


def test_byte_model_ragged_batch_sums_per_request():
    """A ragged batch (prompts of different lengths, a partial last page, per-request retention and windows): the
    cycle's bytes are the sum over requests of the per-request cost model plus each request's generated tokens."""
    import bench
    from oracle import cost_model as cm
    lens, ks, nqs = [4096 + 7, 20000, 65536], [20, 300, 1000], [2, 4, 8]
    hkv, d, k_prop, a, r = 8, 128, 1, 1, 2
    R = len(lens)
    rng = np.random.default_rng(11)
    cap = a + r + max(ks)
    sel = np.zeros((R, hkv, cap), np.int32)
    n_sel = np.zeros((R, hkv), np.int32)
    for i, (L, k) in enumerate(zip(lens, ks)):
        N = (L + 15) // 16
        for h in range(hkv):
            mid = np.sort(rng.choice(np.arange(a, N - r), size=k, replace=False))
            row = np.concatenate([np.arange(a), mid, np.arange(N - r, N)])
            sel[i, h, :row.size] = row
            n_sel[i, h] = row.size
    w = SimpleNamespace(d=d, Hkv=hkv, R=R, k_prop=k_prop, ctx_len=torch.tensor(lens, dtype=torch.int32),
                        seq_len0=torch.tensor(lens, dtype=torch.int32), n_q=torch.tensor(nqs, dtype=torch.int32))
    b = bench.step_bytes(w, None, torch.from_numpy(sel), torch.from_numpy(n_sel))
    kv_tok = d * 2 * 2 * hkv
    total = 0.0
    for i, (L, k, nq) in enumerate(zip(lens, ks, nqs)):
        N = (L + 15) // 16
        last_valid = L - 16 * (N - 1)
        s = (16 * (a + r + k - 1) + last_valid) / L   # every selected page is full except the recent last one
        total += cm.cycle_kv_bytes(k_prop, s, L * kv_tok) + (sum(j + 1 for j in range(k_prop)) + nq) * kv_tok
    assert abs(sum(b["propose"]) + b["verify"] - total) < 1e-6 * total
