"""The bounded waits: a kernel whose wait is never completed gives up, reports bit 8 through kap_device_error, and the
GPU context stays usable for the next call.

Every mbarrier wait of the library's kernels is bounded. The wait here is the same bounded wait, on a barrier that
nothing arrives on, with a short limit, and with no copy or MMA in flight, so giving up leaves nothing pending.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_next_call_succeeds(kap):
    from tests.gpu_helpers import assert_close_attn, run_cycle_and_oracle
    from workloads import make_workload
    assert kap.kap_device_error() == 0
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kap.kap_selftest_wait_timeout(8, 1000, flag)   # 8 polls of at most 1 us: gives up within microseconds
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    assert kap.kap_device_error() == 8               # reported once, then cleared
    assert kap.kap_device_error() == 0
    # a clean cycle right after: selections bit-exact, attention within tolerance, no error
    w = make_workload("llama", device="cuda", scale=1 / 32)
    res = run_cycle_and_oracle(w)
    assert np.array_equal(res["sel_gpu"], res["sel_orc"]) and np.array_equal(res["nsel_gpu"], res["nsel_orc"])
    for i, st in enumerate(res["prop"]):
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, f"propose {i}")
    v = res["ver"]
    assert_close_attn(v["o_gpu"], v["o_orc"], v["lse_gpu"], v["lse_orc"], w.dtype, "verify")
    assert kap.kap_device_error() == 0
