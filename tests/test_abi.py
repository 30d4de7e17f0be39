"""Host-side checks (no GPU): the C-ABI library builds, loads and exports every symbol include/kap.h declares;
the binding's host helpers agree with the pages' definitions."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kap.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kap_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from selected_kv_sparse_gb300 import build as kbuild
    path = kbuild.build()
    import torch  # noqa: F401  (makes the CUDA runtime library resolvable)
    return ctypes.CDLL(path)


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("kap_score_topk", "kap_compile_view", "kap_append_kv", "kap_attn_propose", "kap_attn_verify"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_size_queries(lib):
    lib.kap_status_str.restype = ctypes.c_char_p
    for s in (0, 1, -1, -2, -3, -4, -5):
        assert lib.kap_status_str(s)
    lib.kap_propose_workspace_size.restype = ctypes.c_size_t
    lib.kap_verify_workspace_size.restype = ctypes.c_size_t
    lib.kap_score_workspace_size.restype = ctypes.c_size_t
    assert lib.kap_score_workspace_size(4, 8, 2049) == 4 * 8 * 2049 * 4
    assert lib.kap_propose_workspace_size(4, 8, 32, 128) > 0
    assert lib.kap_verify_workspace_size(4, 8, 32, 128, 4) > 0
    assert lib.kap_verify_workspace_size(0, 8, 32, 128, 4) == 0


def test_null_arguments_are_rejected_without_a_gpu(lib):
    # argument checks run on the host before any CUDA call
    assert lib.kap_attn_propose(None, None, None, None, None, None, None, ctypes.c_size_t(0), None) == -1
    assert lib.kap_score_topk(None, None, None, None, None, None, None, ctypes.c_size_t(0), None) == -1
    assert lib.kap_prior_topk(None, None, 32, 8, None, None, None, None, ctypes.c_size_t(0), None) == -1
    assert lib.kap_accept_commit(None, 1, 128, 1, 5, None, None, None, 3, None, None, None, None,
                                 ctypes.c_size_t(0), None) == -1


def test_parse_ark():
    from selected_kv_sparse_gb300 import parse_ark
    assert parse_ark("A1R2K13") == (1, 2, 13)
    assert parse_ark("A0R0K16") == (0, 0, 16)
    with pytest.raises(ValueError):
        parse_ark("R2K13")


def test_rope_inv_freq_matches_oracle(orc):
    from selected_kv_sparse_gb300 import rope_inv_freq
    for d in (64, 128):
        assert np.array_equal(rope_inv_freq(d).numpy(), orc.inv_freq(d, 1.0e4))


def test_rope_inv_freq_raw_abi(lib, orc):
    """kap_rope_inv_freq through the raw C ABI: bit-identical to the oracle's table for several widths and bases;
    documented argument errors (KAP_EINVAL = -1) for a NULL buffer, odd or non-positive d and a bad theta."""
    f = lib.kap_rope_inv_freq
    f.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    for d in (2, 64, 96, 128, 256):
        for theta in (1.0e4, 5.0e5, 2.0):
            out = np.full(d // 2, np.nan, dtype=np.float32)
            assert f(d, theta, out.ctypes.data) == 0
            assert np.array_equal(out, orc.inv_freq(d, theta)), (d, theta)
    buf = np.zeros(64, dtype=np.float32)
    assert f(128, 1.0e4, None) == -1
    for d, theta in ((0, 1.0e4), (-2, 1.0e4), (63, 1.0e4), (64, 0.0), (64, -1.0), (64, float("nan")),
                     (64, float("inf"))):
        assert f(d, theta, buf.ctypes.data) == -1, (d, theta)


def test_long_spans_recipe():
    import torch
    from workloads.gen import _spans_long
    g = torch.Generator().manual_seed(3)
    sp = _spans_long(g, 8192)
    assert len(sp) == 30
    pages = [(a // 16, n // 16) for a, n in sp]
    assert sum(n for _, n in pages) == 446
    assert all(8 <= n <= 32 for _, n in pages)
    for (a0, n0), (a1, _) in zip(pages, pages[1:]):
        assert a0 + n0 < a1          # non-overlapping and non-adjacent
    assert pages[0][0] >= 1 and pages[-1][0] + pages[-1][1] <= 8188


def test_binding_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors of the header's structs: same size and the same offset for every field, as a C
    compiler lays them out from include/kap.h."""
    import shutil
    import subprocess
    from selected_kv_sparse_gb300 import _binding as kb
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mirrors = {"kap_kv_pool": kb._Pool, "kap_page_map": kb._Map, "kap_access_policy": kb._Policy,
               "kap_view": kb._View, "kap_verify_policy": kb._Verify}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kap.h"', "int main(void) {"]
    for cname, py in mirrors.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
