"""ctypes binding of the C ABI in include/kap.h.

Argument marshalling only: every function takes torch CUDA tensors, checks dtype/shape/contiguity on the host,
passes raw device pointers and the current torch stream to the library, and raises KapError on a non-OK status.
All computation runs in the library's CUDA kernels; there is no CPU path. Loading fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkap.so")

KAP_OK = 0
KAP_FALLBACK_FULL = 1
KAP_BF16 = 0
KAP_F32 = 1
PAGE = 16

_lock = threading.Lock()
_lib = None


class KapError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


class _Pool(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p), ("k_summary", ctypes.c_void_p)]


class _Map(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("ctx_len", ctypes.c_void_p), ("seq_len", ctypes.c_void_p)]


class _Policy(ctypes.Structure):
    _fields_ = [("anchor", ctypes.c_int32), ("recent", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("per_kv_head", ctypes.c_int32), ("cap", ctypes.c_int32), ("per_seq_ark", ctypes.c_void_p)]


class _View(ctypes.Structure):
    _fields_ = [("rows_per_seq", ctypes.c_int32), ("cap", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("logical_page", ctypes.c_void_p), ("n_entries", ctypes.c_void_p), ("n_selected", ctypes.c_void_p),
                ("settled", ctypes.c_int32)]


class _Verify(ctypes.Structure):
    _fields_ = [("max_q", ctypes.c_int32), ("total_q", ctypes.c_int32), ("q_offsets", ctypes.c_void_p),
                ("q_start_pos", ctypes.c_void_p)]


def _declare(lib):
    P, I, Z = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    F = ctypes.c_float
    sig = {
        "kap_build_summaries": ([P, P, P], I),
        "kap_refresh_summaries": ([P, P, P, I, P], I),
        "kap_score_topk": ([P, P, P, P, P, P, P, Z, P], I),
        "kap_prior_topk": ([P, P, I, I, P, P, P, P, Z, P], I),
        "kap_accept_commit": ([P, I, I, I, I, P, P, P, I, P, P, P, P, Z, P], I),
        "kap_materialize_view": ([P, P, P, I, I, P, P, P], I),
        "kap_accept_workspace_size": ([I, I, I], Z),
        "kap_score_workspace_size": ([I, I, I], Z),
        "kap_score_topk_view": ([P, P, P, P, P, P, P, Z, I, P, P, F, P, P, P], I),
        "kap_select_spans": ([P, P, P, P, P, P, P], I),
        "kap_compile_view": ([P, P, P, I, I, I, P, P, F, P, P, P], I),
        "kap_slot_mapping": ([P, P, P, I, P, P, P], I),
        "kap_append_kv": ([P, P, P, P, P, P, I, I, P, P], I),
        "kap_attn_propose": ([P, P, P, P, P, P, P, Z, P], I),
        "kap_append_propose": ([P, P, P, P, P, P, P, P, P, P, Z, P], I),
        "kap_propose_workspace_size": ([I, I, I, I], Z),
        "kap_attn_verify": ([P, P, P, P, P, P, P, Z, P], I),
        "kap_verify_workspace_size": ([I, I, I, I, I], Z),
        "kap_status_str": ([I], ctypes.c_char_p),
        "kap_last_cuda_error": ([], ctypes.c_char_p),
        "kap_device_error": ([P], I),
        "kap_attn_propose_noalloc": ([P, P, P, P, P, P, P], I),
        "kap_noalloc_scratch_bytes": ([], Z),
        "kap_rope_inv_freq": ([I, ctypes.c_double, P], I),
        "kap_selftest_wait_timeout": ([ctypes.c_uint32, ctypes.c_uint32, P, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res


def load():
    """Loads libkap.so (in-tree). Raises if it is missing: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m selected_kv_sparse_gb300.build`")
            import torch.cuda  # noqa: F401  (the CUDA runtime of torch is loaded first and shared)
            lib = ctypes.CDLL(LIB_PATH)
            _declare(lib)
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != KAP_OK:
        lib = load()
        msg = lib.kap_status_str(status).decode()
        if status == -4:
            msg += ": " + lib.kap_last_cuda_error().decode()
        raise KapError(fn, status, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _i32(t, name):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _ptr(t)


# ----------------------------------------------------------------------------------------------- structures
@dataclass
class KVPool:
    """Paged KV pool: k_pages, v_pages [num_pages][Hkv][16][d] (bf16 or fp32); k_summary [num_pages][Hkv][d] fp32."""
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    num_q_heads: int
    k_summary: Optional[torch.Tensor] = None

    def _c(self) -> _Pool:
        k = self.k_pages
        if k.shape != self.v_pages.shape or k.dtype != self.v_pages.dtype or k.dim() != 4 or k.shape[2] != PAGE:
            raise ValueError("k_pages/v_pages must both be [num_pages][Hkv][16][d] of one dtype")
        dt = {torch.bfloat16: KAP_BF16, torch.float32: KAP_F32}.get(k.dtype)
        if dt is None:
            raise TypeError("pool dtype must be bfloat16 or float32")
        if self.k_summary is not None and (self.k_summary.dtype != torch.float32 or
                                           tuple(self.k_summary.shape) != (k.shape[0], k.shape[1], k.shape[3])):
            raise ValueError("k_summary must be fp32 [num_pages][Hkv][d]")
        return _Pool(k.shape[0], PAGE, k.shape[1], self.num_q_heads, k.shape[3], dt, _ptr(k), _ptr(self.v_pages),
                     _ptr(self.k_summary))

    @property
    def dtype(self):
        return self.k_pages.dtype


@dataclass
class PageMap:
    """block_table [R][max_pages] int32; ctx_len, seq_len [R] int32 (device)."""
    block_table: torch.Tensor
    ctx_len: torch.Tensor
    seq_len: Optional[torch.Tensor] = None

    def _c(self) -> _Map:
        bt = self.block_table
        if bt.dim() != 2:
            raise ValueError("block_table must be [R][max_pages]")
        if self.ctx_len.numel() != bt.shape[0] or (self.seq_len is not None and self.seq_len.numel() != bt.shape[0]):
            raise ValueError("ctx_len/seq_len must have R entries")
        return _Map(bt.shape[0], bt.shape[1], _i32(bt, "block_table"), _i32(self.ctx_len, "ctx_len"),
                    _i32(self.seq_len, "seq_len") if self.seq_len is not None else None)


@dataclass
class AccessPolicy:
    """rho_access: A<a>R<r>K<k> split, per-KV-head or shared selection, row capacity, optional per-request ark."""
    anchor: int
    recent: int
    topk: int
    per_kv_head: bool
    cap: int
    per_seq_ark: Optional[torch.Tensor] = None

    def _c(self) -> _Policy:
        return _Policy(self.anchor, self.recent, self.topk, int(self.per_kv_head), self.cap,
                       _i32(self.per_seq_ark, "per_seq_ark") if self.per_seq_ark is not None else None)


def parse_ark(tag: str):
    """'A1R2K125' -> (1, 2, 125) (the KRI page's A<a>R<r>K<k> tag)."""
    import re
    m = re.fullmatch(r"A(\d+)R(\d+)K(\d+)", tag.strip())
    if not m:
        raise ValueError(f"not an A<a>R<r>K<k> tag: {tag!r}")
    return tuple(int(x) for x in m.groups())


@dataclass
class View:
    """Compact selected-KV view buffers (written by kap_compile_view)."""
    rows_per_seq: int
    cap: int
    block_table: torch.Tensor   # [R][rows][cap] int32
    logical_page: torch.Tensor  # [R][rows][cap] int32
    n_entries: torch.Tensor     # [R][rows] int32
    n_selected: torch.Tensor    # [R][rows] int32

    @staticmethod
    def empty(R: int, rows_per_seq: int, cap: int, device) -> "View":
        z = lambda *s: torch.zeros(*s, dtype=torch.int32, device=device)  # noqa: E731
        return View(rows_per_seq, cap, z(R, rows_per_seq, cap), z(R, rows_per_seq, cap), z(R, rows_per_seq),
                    z(R, rows_per_seq))

    def _c(self, settled: bool = False) -> _View:
        return _View(self.rows_per_seq, self.cap, _i32(self.block_table, "view.block_table"),
                     _i32(self.logical_page, "view.logical_page"), _i32(self.n_entries, "view.n_entries"),
                     _i32(self.n_selected, "view.n_selected"), int(bool(settled)))


@dataclass
class VerifyPolicy:
    """rho_verify: request r owns query rows q_offsets[r]..q_offsets[r+1]-1 starting at position q_start_pos[r]."""
    q_offsets: torch.Tensor
    q_start_pos: torch.Tensor
    max_q: int
    total_q: int

    def _c(self) -> _Verify:
        return _Verify(self.max_q, self.total_q, _i32(self.q_offsets, "q_offsets"), _i32(self.q_start_pos, "q_start_pos"))


# ------------------------------------------------------------------------------------------------- calls
def kap_build_summaries(pool: KVPool, pmap: PageMap, stream=None):
    lib = load()
    p, m = pool._c(), pmap._c()
    _check("kap_build_summaries", lib.kap_build_summaries(ctypes.byref(p), ctypes.byref(m), _stream(stream)))


def kap_refresh_summaries(pool: KVPool, pages: torch.Tensor, n_valid: torch.Tensor, stream=None):
    """Recomputes the K summaries of the listed physical pages (int32, device) over their n_valid first tokens."""
    lib = load()
    if pages.shape != n_valid.shape or pages.dim() != 1:
        raise ValueError("pages and n_valid must be 1-D and of equal length")
    p = pool._c()
    _check("kap_refresh_summaries", lib.kap_refresh_summaries(ctypes.byref(p), _i32(pages, "pages"),
                                                              _i32(n_valid, "n_valid"), pages.numel(),
                                                              _stream(stream)))


def kap_score_workspace_size(R: int, rows_per_seq: int, max_pages: int) -> int:
    return int(load().kap_score_workspace_size(R, rows_per_seq, max_pages))


def kap_score_topk(pool: KVPool, pmap: PageMap, q: torch.Tensor, policy: AccessPolicy, sel_ids: torch.Tensor,
                   n_sel: torch.Tensor, workspace: torch.Tensor, stream=None):
    lib = load()
    if q.dtype != pool.dtype:
        raise TypeError("q must have the pool dtype")
    p, m, pol = pool._c(), pmap._c(), policy._c()
    _check("kap_score_topk", lib.kap_score_topk(ctypes.byref(p), ctypes.byref(m), _ptr(q), ctypes.byref(pol),
                                                _i32(sel_ids, "sel_ids"), _i32(n_sel, "n_sel"), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream)))


def kap_prior_topk(pmap: PageMap, affinities: torch.Tensor, policy: AccessPolicy, sel_ids: torch.Tensor,
                   n_sel: torch.Tensor, workspace: torch.Tensor, stream=None):
    """affinities [R][L][H][max_pages] fp32 external prior -> per-request A/R/K selection (one row per request)."""
    lib = load()
    if affinities.dtype != torch.float32 or affinities.dim() != 4 or not affinities.is_contiguous():
        raise TypeError("affinities must be a contiguous fp32 [R][L][H][max_pages] tensor")
    if affinities.shape[0] != pmap.block_table.shape[0] or affinities.shape[3] != pmap.block_table.shape[1]:
        raise ValueError("affinities must be [R][L][H][max_pages] for this page map")
    m, pol = pmap._c(), policy._c()
    _check("kap_prior_topk", lib.kap_prior_topk(ctypes.byref(m), _ptr(affinities), int(affinities.shape[1]),
                                                int(affinities.shape[2]), ctypes.byref(pol),
                                                _i32(sel_ids, "sel_ids"), _i32(n_sel, "n_sel"), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream)))


def kap_materialize_view(pool: KVPool, pmap: PageMap, view: View, ws_first_page: int, ws_pages_per_seq: int,
                         out_view: Optional[View] = None, fallback: Optional[torch.Tensor] = None, stream=None):
    """Copies each view row's selected pages into its request's workspace pages of the pool and points the row
    there (in place when out_view is None)."""
    lib = load()
    out_view = view if out_view is None else out_view
    p, m, v, o = pool._c(), pmap._c(), view._c(), out_view._c()
    _check("kap_materialize_view", lib.kap_materialize_view(
        ctypes.byref(p), ctypes.byref(m), ctypes.byref(v), int(ws_first_page), int(ws_pages_per_seq), ctypes.byref(o),
        _i32(fallback, "fallback") if fallback is not None else None, _stream(stream)))


def kap_accept_workspace_size(num_seqs: int, total_rows: int, vocab: int) -> int:
    return int(load().kap_accept_workspace_size(num_seqs, total_rows, vocab))


def kap_accept_commit(logits: torch.Tensor, window_offsets: torch.Tensor, tokens: torch.Tensor, top_n: int,
                      accepted: torch.Tensor, carry: torch.Tensor, workspace: torch.Tensor,
                      start_pos: Optional[torch.Tensor] = None, seq_len_out: Optional[torch.Tensor] = None,
                      stream=None):
    """Top-n tolerant acceptance of verify windows (logits [total_rows][vocab], bf16 or fp32) and their commit."""
    lib = load()
    if logits.dim() != 2 or not logits.is_contiguous() or logits.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("logits must be a contiguous [total_rows][vocab] bf16 or fp32 tensor")
    dt = KAP_BF16 if logits.dtype == torch.bfloat16 else KAP_F32
    total_rows, vocab = int(logits.shape[0]), int(logits.shape[1])
    R = int(window_offsets.numel()) - 1
    _check("kap_accept_commit", lib.kap_accept_commit(
        _ptr(logits), dt, vocab, R, total_rows, _i32(window_offsets, "window_offsets"), _i32(tokens, "tokens"),
        _i32(start_pos, "start_pos") if start_pos is not None else None, int(top_n), _i32(accepted, "accepted"),
        _i32(carry, "carry"), _i32(seq_len_out, "seq_len_out") if seq_len_out is not None else None,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def kap_score_topk_view(pool: KVPool, pmap: PageMap, q: torch.Tensor, policy: AccessPolicy, sel_ids: torch.Tensor,
                        n_sel: torch.Tensor, workspace: torch.Tensor, horizon_tokens: int, view: View,
                        fallback: Optional[torch.Tensor] = None, s_max: float = 1.0,
                        slot_out: Optional[torch.Tensor] = None, pos_out: Optional[torch.Tensor] = None,
                        stream=None):
    """kap_score_topk and kap_compile_view in one call (the top-K kernel compiles each row's view)."""
    lib = load()
    if q.dtype != pool.dtype:
        raise TypeError("q must have the pool dtype")
    if slot_out is not None and (slot_out.dtype != torch.int64 or slot_out.numel() < pmap.block_table.shape[0] *
                                 horizon_tokens):
        raise ValueError("slot_out must be int64 with R * horizon_tokens elements")
    p, m, pol, v = pool._c(), pmap._c(), policy._c(), view._c()
    _check("kap_score_topk_view", lib.kap_score_topk_view(
        ctypes.byref(p), ctypes.byref(m), _ptr(q), ctypes.byref(pol), _i32(sel_ids, "sel_ids"), _i32(n_sel, "n_sel"),
        _ptr(workspace), workspace.numel() * workspace.element_size(), horizon_tokens, ctypes.byref(v),
        _i32(fallback, "fallback") if fallback is not None else None, float(s_max), _ptr(slot_out),
        _i32(pos_out, "pos_out") if pos_out is not None else None, _stream(stream)))


def kap_select_spans(pmap: PageMap, spans: torch.Tensor, span_offsets: torch.Tensor, policy: AccessPolicy,
                     sel_ids: torch.Tensor, n_sel: torch.Tensor, stream=None):
    lib = load()
    m, pol = pmap._c(), policy._c()
    _check("kap_select_spans", lib.kap_select_spans(ctypes.byref(m), _i32(spans, "spans"),
                                                    _i32(span_offsets, "span_offsets"), ctypes.byref(pol),
                                                    _i32(sel_ids, "sel_ids"), _i32(n_sel, "n_sel"), _stream(stream)))


def kap_compile_view(pmap: PageMap, sel_ids: torch.Tensor, n_sel: torch.Tensor, horizon_tokens: int, view: View,
                     fallback: Optional[torch.Tensor] = None, s_max: float = 1.0,
                     slot_out: Optional[torch.Tensor] = None, pos_out: Optional[torch.Tensor] = None, stream=None):
    """Compact view; optionally also the slot mapping [R][horizon_tokens] of the tokens the cycle appends."""
    lib = load()
    if sel_ids.dim() != 3:
        raise ValueError("sel_ids must be [R][rows][cap]")
    if slot_out is not None and (slot_out.dtype != torch.int64 or slot_out.numel() < pmap.block_table.shape[0] *
                                 horizon_tokens):
        raise ValueError("slot_out must be int64 with R * horizon_tokens elements")
    m, v = pmap._c(), view._c()
    _check("kap_compile_view", lib.kap_compile_view(ctypes.byref(m), _i32(sel_ids, "sel_ids"), _i32(n_sel, "n_sel"),
                                                    sel_ids.shape[1], sel_ids.shape[2], horizon_tokens,
                                                    ctypes.byref(v),
                                                    _i32(fallback, "fallback") if fallback is not None else None,
                                                    float(s_max), _ptr(slot_out),
                                                    _i32(pos_out, "pos_out") if pos_out is not None else None,
                                                    _stream(stream)))


def kap_slot_mapping(pmap: PageMap, tok_offsets: torch.Tensor, start_pos: torch.Tensor, slot_out: torch.Tensor,
                     pos_out: Optional[torch.Tensor] = None, stream=None):
    lib = load()
    if slot_out.dtype != torch.int64:
        raise TypeError("slot_out must be int64")
    m = pmap._c()
    _check("kap_slot_mapping", lib.kap_slot_mapping(ctypes.byref(m), _i32(tok_offsets, "tok_offsets"),
                                                    _i32(start_pos, "start_pos"), slot_out.numel(), _ptr(slot_out),
                                                    _i32(pos_out, "pos_out") if pos_out is not None else None,
                                                    _stream(stream)))


def kap_append_kv(pool: KVPool, k_new: torch.Tensor, v_new: torch.Tensor, q_inout: Optional[torch.Tensor],
                  pos: torch.Tensor, slots: torch.Tensor, inv_freq: torch.Tensor, num_tokens: Optional[int] = None,
                  tok_stride: int = 1, stream=None):
    lib = load()
    if k_new.dtype != pool.dtype or v_new.dtype != pool.dtype or (q_inout is not None and q_inout.dtype != pool.dtype):
        raise TypeError("k_new, v_new and q must have the pool dtype")
    if slots.dtype != torch.int64 or inv_freq.dtype != torch.float32:
        raise TypeError("slots must be int64 and inv_freq fp32")
    T = k_new.shape[0] if num_tokens is None else num_tokens
    p = pool._c()
    _check("kap_append_kv", lib.kap_append_kv(ctypes.byref(p), _ptr(k_new), _ptr(v_new), _ptr(q_inout),
                                              _i32(pos, "pos"), _ptr(slots), T, tok_stride, _ptr(inv_freq),
                                              _stream(stream)))


def kap_propose_workspace_size(R: int, hkv: int, hq: int, d: int) -> int:
    return int(load().kap_propose_workspace_size(R, hkv, hq, d))


def kap_attn_propose(pool: KVPool, pmap: PageMap, view: View, q: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                     workspace: torch.Tensor, stream=None, settled: bool = False):
    """settled: the caller's promise that the view, the page map and the prompt tokens were written before the
    kernel launched just ahead of this call on the stream (kap_view.settled)."""
    lib = load()
    if q.dtype != pool.dtype or out.dtype != pool.dtype or lse.dtype != torch.float32:
        raise TypeError("q/out must have the pool dtype and lse fp32")
    p, m, v = pool._c(), pmap._c(), view._c(settled)
    _check("kap_attn_propose", lib.kap_attn_propose(ctypes.byref(p), ctypes.byref(m), ctypes.byref(v), _ptr(q),
                                                    _ptr(out), _ptr(lse), _ptr(workspace),
                                                    workspace.numel() * workspace.element_size(), _stream(stream)))


def kap_append_propose(pool: KVPool, pmap: PageMap, view: View, q: torch.Tensor, k_new: torch.Tensor,
                       v_new: torch.Tensor, inv_freq: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                       workspace: torch.Tensor, stream=None, settled: bool = False):
    """One proposal step with the step token's KV append fused in: the token of request r sits at seq_len[r]-1;
    q holds the step's queries before RoPE (read only). settled: as for kap_attn_propose."""
    lib = load()
    if any(t.dtype != pool.dtype for t in (q, k_new, v_new, out)) or lse.dtype != torch.float32:
        raise TypeError("q, k_new, v_new and out must have the pool dtype and lse fp32")
    if inv_freq.dtype != torch.float32:
        raise TypeError("inv_freq must be fp32")
    p, m, v = pool._c(), pmap._c(), view._c(settled)
    _check("kap_append_propose", lib.kap_append_propose(ctypes.byref(p), ctypes.byref(m), ctypes.byref(v), _ptr(q),
                                                        _ptr(k_new), _ptr(v_new), _ptr(inv_freq), _ptr(out),
                                                        _ptr(lse), _ptr(workspace),
                                                        workspace.numel() * workspace.element_size(),
                                                        _stream(stream)))


def kap_attn_propose_noalloc(pool: KVPool, pmap: PageMap, view: View, q: torch.Tensor, out: torch.Tensor,
                             lse: torch.Tensor, stream=None):
    """kap_attn_propose without a workspace argument: the library's own fixed scratch array is used instead (for
    callers that may not allocate device memory). Calls that overlap on the GPU share that scratch and race."""
    lib = load()
    if q.dtype != pool.dtype or out.dtype != pool.dtype or lse.dtype != torch.float32:
        raise TypeError("q/out must have the pool dtype and lse fp32")
    p, m, v = pool._c(), pmap._c(), view._c()
    _check("kap_attn_propose_noalloc", lib.kap_attn_propose_noalloc(ctypes.byref(p), ctypes.byref(m), ctypes.byref(v),
                                                                    _ptr(q), _ptr(out), _ptr(lse), _stream(stream)))


def kap_noalloc_scratch_bytes() -> int:
    return int(load().kap_noalloc_scratch_bytes())


def kap_verify_workspace_size(R: int, hkv: int, hq: int, d: int, max_q: int) -> int:
    return int(load().kap_verify_workspace_size(R, hkv, hq, d, max_q))


def kap_attn_verify(pool: KVPool, pmap: PageMap, vp: VerifyPolicy, q: torch.Tensor, out: torch.Tensor,
                    lse: torch.Tensor, workspace: torch.Tensor, stream=None):
    lib = load()
    if q.dtype != pool.dtype or out.dtype != pool.dtype or lse.dtype != torch.float32:
        raise TypeError("q/out must have the pool dtype and lse fp32")
    p, m, v = pool._c(), pmap._c(), vp._c()
    _check("kap_attn_verify", lib.kap_attn_verify(ctypes.byref(p), ctypes.byref(m), ctypes.byref(v), _ptr(q),
                                                  _ptr(out), _ptr(lse), _ptr(workspace),
                                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def kap_selftest_wait_timeout(polls: int, suspend_ns: int, timed_out: torch.Tensor, stream=None):
    """Runs the library's bounded mbarrier wait on a barrier that nothing completes (see kap.h); timed_out is a
    one-element int32 CUDA tensor that receives 1 when the wait gave up."""
    if timed_out.dtype != torch.int32 or not timed_out.is_cuda or timed_out.numel() < 1:
        raise ValueError("timed_out must be an int32 CUDA tensor")
    _check("kap_selftest_wait_timeout",
           load().kap_selftest_wait_timeout(int(polls), int(suspend_ns), _ptr(timed_out), _stream(stream)))


def kap_device_error() -> int:
    lib = load()
    code = ctypes.c_int32(0)
    _check("kap_device_error", lib.kap_device_error(ctypes.byref(code)))
    return int(code.value)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled device workspace of at least nbytes (counters inside must start at zero)."""
    return torch.zeros(max(1, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)


def rope_inv_freq(d: int, theta: float = 1.0e4, device="cpu") -> torch.Tensor:
    """RoPE inverse frequencies theta^(-2i/d), i < d/2, from the library (kap_rope_inv_freq: fp64, rounded once to
    fp32), as a tensor on `device`."""
    out = torch.empty(d // 2, dtype=torch.float32)
    _check("kap_rope_inv_freq", load().kap_rope_inv_freq(int(d), float(theta), ctypes.c_void_p(out.data_ptr())))
    return out.to(device)
