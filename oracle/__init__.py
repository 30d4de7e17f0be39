"""CPU oracle of the selected-KV sparse decode hot path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this package.
The product library (``selected_kv_sparse_gb300``) never imports it and has no fallback to it.

The arithmetic lives in ``kap_oracle.cpp`` (plain C++, fp64 attention); this module compiles it with g++ and
marshals numpy arrays to it. ``cost_model`` holds the pages' memory-traffic cost model. No function here shares
code with the CUDA library: they meet only on the seeded inputs of ``workloads``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kap_oracle.cpp")
_LIB = os.path.join(_HERE, "libkap_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE = 16


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source (g++, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_build_summaries.argtypes = [P, I, I, I, P, I, I, P, P]
            lib.orc_build_summaries.restype = I
            lib.orc_dot_fixed_order.argtypes = [P, P, I]
            lib.orc_dot_fixed_order.restype = ctypes.c_float
            lib.orc_scores.argtypes = [P, P, I, I, I, P, I, I, P, I, P, P]
            lib.orc_scores.restype = I
            lib.orc_topk_ark.argtypes = [P, I, I, I, I, P]
            lib.orc_topk_ark.restype = I
            lib.orc_prior_scores.argtypes = [P, I, I, I, P]
            lib.orc_prior_scores.restype = I
            lib.orc_accept_commit.argtypes = [P, I, I, P, I, I, P, P, P]
            lib.orc_accept_commit.restype = I
            lib.orc_materialize_row.argtypes = [P, P, I, I, I, I, I, P, P, P]
            lib.orc_materialize_row.restype = I
            lib.orc_select_spans.argtypes = [I, P, I, I, I, P]
            lib.orc_select_spans.restype = I
            lib.orc_compile_view_row.argtypes = [P, I, I, I, P, I, P, P, P]
            lib.orc_compile_view_row.restype = I
            lib.orc_slot.argtypes = [P, I, I]
            lib.orc_slot.restype = ctypes.c_int64
            lib.orc_inv_freq.argtypes = [I, ctypes.c_double, P]
            lib.orc_inv_freq.restype = None
            lib.orc_rope.argtypes = [P, I, I, I, P, P, P]
            lib.orc_rope.restype = None
            lib.orc_attn_propose.argtypes = [P, P, P, I, I, I, I, P, I, I, P, P, P, P, I, I, P, P, I]
            lib.orc_attn_propose.restype = I
            lib.orc_attn_verify.argtypes = [P, P, P, I, I, I, I, P, I, I, P, P, P, P, I]
            lib.orc_attn_verify.restype = I
            lib.orc_hardware_threads.argtypes = []
            lib.orc_hardware_threads.restype = I
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def build_summaries(K, block_table, ctx_len):
    """Block-mean K per (page, KV head) for every prompt page of every request. K: [P][Hkv][16][d]."""
    K = _f32(K)
    P, hkv, _, d = K.shape
    bt = _i32(block_table)
    cl = _i32(ctx_len)
    S = np.zeros((P, hkv, d), dtype=np.float32)
    rc = _load().orc_build_summaries(_p(K), P, hkv, d, _p(bt), bt.shape[0], bt.shape[1], _p(cl), _p(S))
    if rc != 0:
        raise ValueError("block table references a page outside the pool")
    return S


def dot_fixed_order(a, b) -> np.float32:
    a, b = _f32(a), _f32(b)
    return np.float32(_load().orc_dot_fixed_order(_p(a), _p(b), a.shape[0]))


def scores(q, S, block_table, ctx_len, per_head: bool):
    """Page scores (fp32 fixed order) and their fp64 values. q: [R][Hq][d]. Returns [R][rows][max_pages]."""
    q, S = _f32(q), _f32(S)
    R, hq, d = q.shape
    hkv = S.shape[1]
    bt, cl = _i32(block_table), _i32(ctx_len)
    rows = hkv if per_head else 1
    out = np.full((R, rows, bt.shape[1]), np.nan, dtype=np.float32)
    out64 = np.full((R, rows, bt.shape[1]), np.nan, dtype=np.float64)
    _load().orc_scores(_p(q), _p(S), hq, hkv, d, _p(bt), R, bt.shape[1], _p(cl), int(per_head), _p(out), _p(out64))
    return out, out64


def topk_ark(scores_row, N: int, a: int, r: int, k: int):
    s = _f32(scores_row[:N])
    out = np.zeros(max(N, 1), dtype=np.int32)
    n = _load().orc_topk_ark(_p(s), N, a, r, k, _p(out))
    return out[:n].copy()


def prior_scores(aff):
    """aff [L][H][N] external-prior block affinities of one request -> mean-pooled scores [N] (fp32, fixed order)."""
    a = _f32(aff)
    L, H, N = a.shape
    out = np.zeros(N, dtype=np.float32)
    if _load().orc_prior_scores(_p(a), L, H, N, _p(out)) != 0:
        raise ValueError("bad prior shape")
    return out


def accept_commit(logits, tokens, top_n: int, start_pos: int):
    """One verify window: logits [rows][V], tokens [rows] (carry, then proposals) -> (m, next carry, seq_len)."""
    lg = _f32(logits)
    tk = _i32(tokens)
    rows, V = lg.shape
    assert tk.shape == (rows,)
    m, c, sl = (np.zeros(1, np.int32) for _ in range(3))
    if _load().orc_accept_commit(_p(lg), rows, V, _p(tk), top_n, start_pos, _p(m), _p(c), _p(sl)) != 0:
        raise ValueError("bad window")
    return int(m[0]), int(c[0]), int(sl[0])


def materialize_row(bt_row, lp_row, n_entries: int, n_selected: int, ctx_len: int, ws_base: int, ws_pages: int):
    """One view row into its workspace -> (new row [n_entries], [(src page, dst page)], fits)."""
    bt = _i32(np.asarray(bt_row)[:max(n_entries, 1)])
    lp = _i32(np.asarray(lp_row)[:max(n_entries, 1)])
    out = np.zeros(max(n_entries, 1), np.int32)
    src = np.zeros(max(n_selected, 1), np.int32)
    dst = np.zeros(max(n_selected, 1), np.int32)
    n = _load().orc_materialize_row(_p(bt), _p(lp), n_entries, n_selected, ctx_len, ws_base, ws_pages, _p(out),
                                    _p(src), _p(dst))
    pairs = [] if n < 0 else list(zip(src[:n].tolist(), dst[:n].tolist()))
    return out[:n_entries], pairs, n >= 0


def select_spans(N: int, spans, a: int, r: int):
    sp = _i32(np.asarray(spans, dtype=np.int32).reshape(-1, 2))
    out = np.zeros(max(N, 1), dtype=np.int32)
    n = _load().orc_select_spans(N, _p(sp), sp.shape[0], a, r, _p(out))
    return out[:n].copy()


def compile_view_row(block_table_row, ctx_len: int, seq_len: int, horizon: int, sel):
    bt = _i32(block_table_row)
    sel = _i32(sel)
    cap = len(sel) + (seq_len + horizon) // PAGE + 2 - ctx_len // PAGE
    cap = max(cap, 1)
    cbt = np.zeros(cap, dtype=np.int32)
    clog = np.zeros(cap, dtype=np.int32)
    nsel = np.zeros(1, dtype=np.int32)
    n = _load().orc_compile_view_row(_p(bt), ctx_len, seq_len, horizon, _p(sel), len(sel), _p(cbt), _p(clog),
                                     _p(nsel))
    return cbt[:n].copy(), clog[:n].copy(), int(nsel[0])


def slot(block_table_row, pos: int) -> int:
    bt = _i32(block_table_row)
    return int(_load().orc_slot(_p(bt), bt.shape[0], int(pos)))


def inv_freq(d: int, theta: float = 1.0e4):
    out = np.zeros(d // 2, dtype=np.float32)
    _load().orc_inv_freq(d, float(theta), _p(out))
    return out


def rope(x, pos, inv_freq_f32):
    """RoPE of x [T][H][d] at positions pos [T], fp64 result."""
    x = _f32(x)
    T, H, d = x.shape
    pos = _i32(pos)
    f = _f32(inv_freq_f32)
    out = np.zeros((T, H, d), dtype=np.float64)
    _load().orc_rope(_p(x), T, H, d, _p(pos), _p(f), _p(out))
    return out


def attn_propose(q, K, V, block_table, ctx_len, seq_len, sel, nsel, nthreads: int = 1):
    """Proposal attention by enumeration. q [R][Hq][d]; K, V [P][Hkv][16][d]; sel [R][rows][cap]; nsel [R][rows]."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    R, hq, d = q.shape
    P, hkv = K.shape[0], K.shape[1]
    bt, cl, sl = _i32(block_table), _i32(ctx_len), _i32(seq_len)
    sel, nsel = _i32(sel), _i32(nsel)
    rows, cap = sel.shape[1], sel.shape[2]
    out = np.zeros((R, hq, d), dtype=np.float64)
    lse = np.zeros((R, hq), dtype=np.float64)
    rc = _load().orc_attn_propose(_p(q), _p(K), _p(V), P, hq, hkv, d, _p(bt), R, bt.shape[1], _p(cl), _p(sl),
                                  _p(sel), _p(nsel), rows, cap, _p(out), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("block table references a page outside the pool")
    return out, lse


def attn_verify(q, K, V, block_table, q_offsets, q_start, nthreads: int = 1):
    """Verification attention by enumeration. q [total_q][Hq][d]; rows of request r are q_offsets[r]..[r+1]."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    tq, hq, d = q.shape
    P, hkv = K.shape[0], K.shape[1]
    bt, qo, qs = _i32(block_table), _i32(q_offsets), _i32(q_start)
    R = bt.shape[0]
    out = np.zeros((tq, hq, d), dtype=np.float64)
    lse = np.zeros((tq, hq), dtype=np.float64)
    rc = _load().orc_attn_verify(_p(q), _p(K), _p(V), P, hq, hkv, d, _p(bt), R, bt.shape[1], _p(qo), _p(qs),
                                 _p(out), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("block table references a page outside the pool")
    return out, lse
