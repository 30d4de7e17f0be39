"""GB300-native selected-KV sparse decode hot path.

Page scoring and A<a>R<r>K<k> top-K over a K-summary cache, compact selected-KV views with slot mappings that keep
logical positions, RoPE'd KV append, paged GQA proposal attention (q = 1) over the selected pages, and paged causal
verification attention (q = n) over the full block table. Every step is a hand-written sm_103a CUDA kernel behind
the C ABI in include/kap.h; this package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    AccessPolicy, KapError, KVPool, PageMap, VerifyPolicy, View, kap_append_kv, kap_attn_propose, kap_attn_verify,
    kap_build_summaries, kap_compile_view, kap_device_error, kap_propose_workspace_size, kap_score_topk,
    kap_score_workspace_size, kap_select_spans, kap_slot_mapping, kap_verify_workspace_size, load, parse_ark,
    rope_inv_freq, workspace, LIB_PATH,
)
from ._binding import kap_append_propose, kap_attn_propose_noalloc, kap_noalloc_scratch_bytes  # noqa: F401
from ._binding import kap_accept_commit, kap_accept_workspace_size, kap_materialize_view, kap_prior_topk  # noqa: F401
from ._binding import kap_refresh_summaries, kap_score_topk_view, kap_selftest_wait_timeout  # noqa: F401
from .pipeline import DecodeCycle, DecodeLoop, SideFlowDecode  # noqa: F401
