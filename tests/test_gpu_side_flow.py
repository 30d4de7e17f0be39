"""EarlySelectKV side flow: routing of layer l + 1 on a second stream during layer l's step (through the C ABI).

The overlapped schedule runs the same calls as the sequential one, so every layer's selection, view and proposal
output must equal, bit for bit, those of a cycle whose proposal the oracle checks; the schedule must also survive
CUDA-graph capture across the two streams.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LAYERS = 3


def _layers(kap, batch, scale):
    from tests.gpu_helpers import make_cycle
    from workloads import make_workload
    out = []
    for l in range(LAYERS):
        w = make_workload("early", device="cuda", scale=scale, batch=batch, seed_offset=l, poison=False)
        pool, cyc = make_cycle(w)
        kap.kap_build_summaries(pool, kap.PageMap(w.block_table, w.ctx_len, w.seq_len0))
        out.append((w, cyc))
    return out


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


# reduced prompts eager and captured; the full-size prompts (40960 tokens, batch 8) as the benchmark runs them, captured
@pytest.mark.parametrize("batch,scale,graph", [(1, 1 / 16, False), (1, 1 / 16, True), (3, 1 / 16, False),
                                               (3, 1 / 16, True), (8, 1.0, True)])
def test_side_flow_equals_checked_cycles(kap, batch, scale, graph):
    from selected_kv_sparse_gb300.pipeline import SideFlowDecode
    from tests.gpu_helpers import assert_close_attn, run_cycle_and_oracle
    from workloads import make_workload
    # reference: each layer's full cycle against the oracle (its first proposal step is the decode step)
    ref = []
    for l in range(LAYERS):
        w = make_workload("early", device="cuda", scale=scale, batch=batch, seed_offset=l, poison=False)
        res = run_cycle_and_oracle(w, nthreads=16)
        assert np.array_equal(res["sel_gpu"], res["sel_orc"])
        st = res["prop"][0]
        assert_close_attn(st["o_gpu"], st["o_orc"], st["lse_gpu"], st["lse_orc"], w.dtype, "propose")
        ref.append(res["cycle"])
    # the side flow on fresh copies of the same layers
    layers = _layers(kap, batch, scale)
    flow = SideFlowDecode([c for _, c in layers])
    args = ([w.q_route for w, _ in layers], [w.q_prop[0] for w, _ in layers],
            [w.k_new_prop[0] for w, _ in layers], [w.v_new_prop[0] for w, _ in layers])
    if graph:
        flow.step(*args)   # eager once (kernel attributes, stream set-up), then capture and replay
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            flow.step(*args)
        for c in flow.cycles:
            c.o_prop.zero_()
        g.replay()
    else:
        flow.step(*args)
    torch.cuda.synchronize()
    for l, ((w, c), r) in enumerate(zip(layers, ref)):
        assert torch.equal(c.sel_ids, r.sel_ids) and torch.equal(c.n_sel, r.n_sel), l
        assert torch.equal(c.view.block_table, r.view.block_table), l
        assert torch.equal(_bits(c.o_prop[0]), _bits(r.o_prop[0])), l
        assert torch.equal(_bits(c.lse_prop[0]), _bits(r.lse_prop[0])), l
    assert kap.kap_device_error() == 0
