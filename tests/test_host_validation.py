"""Host-side argument checks of the C ABI: each call must return its documented error code before any CUDA call.

The structs carry placeholder addresses that nothing dereferences when the checks work. These tests run only on a
machine without a GPU, so that a check that stopped working could never launch a kernel on such addresses.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host checks run where no kernel can launch")

KAP_EINVAL, KAP_ESHAPE, KAP_ECAPACITY, KAP_EUNSUPPORTED = -1, -2, -3, -5
ADDR = 0x10000  # a placeholder, 16-byte aligned, never dereferenced
Z = ctypes.c_size_t


@pytest.fixture(scope="module")
def abi():
    import selected_kv_sparse_gb300._binding as b
    return b, b.load()


def _pool(b, P=8, hkv=2, hq=8, d=64, dtype=0):
    return b._Pool(P, 16, hkv, hq, d, dtype, ADDR, ADDR, ADDR)


def _map(b, R=2, max_pages=4):
    return b._Map(R, max_pages, ADDR, ADDR, ADDR)


def _ref(x):
    return ctypes.byref(x)


def test_pool_shapes_are_checked(abi):
    b, lib = abi
    pol = b._Policy(1, 1, 1, 1, 4, None)
    args = lambda pool: (_ref(pool), _ref(_map(b)), ctypes.c_void_p(ADDR), _ref(pol), ctypes.c_void_p(ADDR),
                         ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR), Z(1 << 20), None)  # noqa: E731
    assert lib.kap_score_topk(*args(_pool(b, d=96))) == KAP_EUNSUPPORTED           # head_dim 96
    assert lib.kap_score_topk(*args(_pool(b, hkv=2, hq=32))) == KAP_EUNSUPPORTED   # G = 16
    assert lib.kap_score_topk(*args(_pool(b, hkv=2, hq=7))) == KAP_ESHAPE          # 7 query heads on 2 KV heads
    assert lib.kap_score_topk(*args(_pool(b, dtype=7))) == KAP_EUNSUPPORTED        # no such dtype
    bad = _pool(b)
    bad.page_size = 32
    assert lib.kap_score_topk(*args(bad)) == KAP_EUNSUPPORTED                      # pages of 32 tokens


def test_capacities_are_checked(abi):
    b, lib = abi
    ws_need = lib.kap_score_workspace_size(2, 2, 4)
    call = lambda pol, mp, ws: lib.kap_score_topk(  # noqa: E731
        _ref(_pool(b)), _ref(_map(b, max_pages=mp)), ctypes.c_void_p(ADDR), _ref(pol), ctypes.c_void_p(ADDR),
        ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR), Z(ws), None)
    # a + r + k over the row capacity while the rows hold more pages than that
    assert call(b._Policy(1, 1, 5, 1, 3, None), 16, 1 << 20) == KAP_ECAPACITY
    # a score workspace one byte short
    assert call(b._Policy(1, 1, 1, 1, 4, None), 4, ws_need - 1) == KAP_ECAPACITY
    # more (request, KV head) rows than the scoring grid can hold: 32768 requests x 2 KV heads
    assert lib.kap_score_topk(_ref(_pool(b)), _ref(_map(b, R=32768)), ctypes.c_void_p(ADDR),
                              _ref(b._Policy(1, 1, 1, 1, 4, None)), ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR),
                              ctypes.c_void_p(ADDR), Z(1 << 40), None) == KAP_EUNSUPPORTED
    # a view too small for the selection plus the horizon's tail pages: cap 4 + ceil(16/16) + 1 > 5
    view = b._View(2, 5, ADDR, ADDR, ADDR, ADDR, 0)
    assert lib.kap_compile_view(_ref(_map(b)), ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR), 2, 4, 16, _ref(view),
                                None, ctypes.c_float(1.0), None, None, None) == KAP_ECAPACITY


def test_misaligned_query_is_rejected(abi):
    b, lib = abi
    pol = b._Policy(1, 1, 1, 1, 4, None)
    assert lib.kap_score_topk(_ref(_pool(b)), _ref(_map(b)), ctypes.c_void_p(ADDR + 2), _ref(pol),
                              ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR), ctypes.c_void_p(ADDR), Z(1 << 20),
                              None) == KAP_EINVAL


def test_next_row_entry_points_check_their_arguments(abi):
    b, lib = abi
    P = ctypes.c_void_p(ADDR)
    # external prior: per-KV-head rows (the connector selects per request); L*H over 2048
    assert lib.kap_prior_topk(_ref(_map(b)), P, 4, 2, _ref(b._Policy(1, 1, 1, 1, 4, None)), P, P, P, Z(1 << 20),
                              None) == KAP_EINVAL
    assert lib.kap_prior_topk(_ref(_map(b)), P, 64, 33, _ref(b._Policy(1, 1, 1, 0, 4, None)), P, P, P, Z(1 << 20),
                              None) == KAP_EINVAL
    # acceptance: fewer rows than requests; no such dtype; a workspace too small
    assert lib.kap_accept_commit(P, 1, 100, 2, 1, P, P, P, 3, P, P, None, P, Z(1 << 20), None) == KAP_EINVAL
    assert lib.kap_accept_commit(P, 5, 100, 2, 4, P, P, P, 3, P, P, None, P, Z(1 << 20), None) == KAP_EUNSUPPORTED
    assert lib.kap_accept_commit(P, 1, 100, 2, 4, P, P, P, 3, P, P, None, P, Z(8), None) == KAP_ECAPACITY
    # materialisation: workspace pages past the pool; rows that are neither 1 nor Hkv
    v = b._View(2, 6, ADDR, ADDR, ADDR, ADDR, 0)
    assert lib.kap_materialize_view(_ref(_pool(b, P=8)), _ref(_map(b)), _ref(v), 6, 2, _ref(v), None, None) == \
        KAP_ECAPACITY
    v3 = b._View(3, 6, ADDR, ADDR, ADDR, ADDR, 0)
    assert lib.kap_materialize_view(_ref(_pool(b, P=8)), _ref(_map(b)), _ref(v3), 0, 2, _ref(v3), None, None) == \
        KAP_ESHAPE


def test_refresh_checks_its_arguments(abi):
    b, lib = abi
    P = ctypes.c_void_p(ADDR)
    assert lib.kap_refresh_summaries(_ref(_pool(b)), P, P, -1, None) == KAP_EINVAL      # negative count
    assert lib.kap_refresh_summaries(_ref(_pool(b)), None, P, 3, None) == KAP_EINVAL    # no page list
    assert lib.kap_refresh_summaries(_ref(_pool(b)), P, None, 3, None) == KAP_EINVAL    # no counts
    assert lib.kap_refresh_summaries(_ref(_pool(b)), P, P, 0, None) == 0               # nothing listed: no launch
    bad = _pool(b)
    bad.k_summary = None
    assert lib.kap_refresh_summaries(_ref(bad), P, P, 3, None) == KAP_EINVAL            # pool without summaries
    assert lib.kap_refresh_summaries(_ref(_pool(b, d=96)), P, P, 3, None) == KAP_EUNSUPPORTED


def test_wait_check_rejects_out_of_range_limits(abi):
    b, lib = abi
    P = ctypes.c_void_p(ADDR)
    assert lib.kap_selftest_wait_timeout(0, 1000, P, None) == KAP_EINVAL          # no poll
    assert lib.kap_selftest_wait_timeout(1025, 1000, P, None) == KAP_EINVAL       # more polls than a kernel's wait
    assert lib.kap_selftest_wait_timeout(8, 0, P, None) == KAP_EINVAL             # no suspension
    assert lib.kap_selftest_wait_timeout(8, (1 << 20) + 1, P, None) == KAP_EINVAL  # longer than a kernel's poll
    assert lib.kap_selftest_wait_timeout(8, 1000, None, None) == KAP_EINVAL       # nowhere to report
