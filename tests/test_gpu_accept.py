"""Top-n tolerant acceptance and commit of verify windows (KAP paper, verifier) through the C ABI against the oracle.

Accepted counts, next carries and committed lengths are integers decided by comparisons of the same logits on both
sides, so they must match exactly.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="llama", n_q=5, vocab=128256, top_n=3),                      # carry + 4 proposals, Llama-3 vocabulary
    dict(name="llama", n_q=5, vocab=128256, top_n=3, dtype="bf16"),
    dict(name="llama", n_q=5, vocab=1000, top_n=1),                        # greedy exact match
    dict(name="llama", n_q=9, vocab=4097, top_n=3, ties=True),             # tied logits, a ragged last chunk
    dict(name="mixed", vocab=32000, top_n=3, accept=0.6),                  # windows of 2, 4 or 8 rows per request
    dict(name="llama", n_q=1, vocab=5000, top_n=3),                        # a window that is the carry alone
]


def _id(c):
    return "-".join(f"{k}={v}" for k, v in c.items())


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_accept_commit_matches_oracle(kap, case):
    import oracle
    from workloads import make_verify_logits, make_workload
    w = make_workload(case["name"], device="cpu", scale=1 / 32, n_q_override=case.get("n_q"), poison=False)
    dt = torch.bfloat16 if case.get("dtype") == "bf16" else torch.float32
    lg, tok, off = make_verify_logits(w, case["vocab"], accept=case.get("accept", 0.9), dtype=dt,
                                      ties=case.get("ties", False))
    R = w.R
    rows = int(off[-1])
    start = (w.ctx_len + 3).to(torch.int32)   # the carry's position: any start works, the commit adds 1 + m
    dev = "cuda"
    acc = torch.full((R,), -1, dtype=torch.int32, device=dev)
    car = torch.full((R,), -1, dtype=torch.int32, device=dev)
    sl = torch.full((R,), -1, dtype=torch.int32, device=dev)
    ws = torch.zeros(kap.kap_accept_workspace_size(R, rows, case["vocab"]), dtype=torch.uint8, device=dev)
    lg_d, tok_d, off_d, start_d = lg.to(dev), tok.to(dev), off.to(dev), start.to(dev)
    for _ in range(2):   # twice: the call leaves its counters at zero for the next one
        kap.kap_accept_commit(lg_d, off_d, tok_d, case["top_n"], acc, car, ws, start_pos=start_d, seq_len_out=sl)
        torch.cuda.synchronize()
        lg32 = lg.to(torch.float32).numpy()
        for r in range(R):
            a, b = int(off[r]), int(off[r + 1])
            m, c, s = oracle.accept_commit(lg32[a:b], tok[a:b].numpy(), case["top_n"], int(start[r]))
            assert (int(acc[r]), int(car[r]), int(sl[r])) == (m, c, s), f"request {r}"
    assert kap.kap_device_error() == 0
    if case.get("accept", 0.9) >= 0.9 and case["top_n"] == 3 and case.get("n_q", 2) > 1:
        # the planted decisions show: most proposals pass
        assert float(acc.float().mean()) > 0.5 * (float(w.n_q.float().mean()) - 1)
