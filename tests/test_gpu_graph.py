"""One step of the path (schedule rebuild, key statistics with a caller
workspace, attention) captured in a CUDA graph and replayed: every call is
asynchronous and allocates nothing while it runs, so the step can be captured
once and launched as one graph, and each replay writes the same bytes as the
eager calls, also after the inputs change in place. The second geometry's
attention call is two launches, the gathered tiles a programmatic dependent of
the tile pairs, which the capture keeps as such."""
import pytest
import torch

import block_sparse_video_frame_gb300 as vd
from block_sparse_video_frame_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    configs.SMALL.with_(name="small_graph", H=4, outlier_heads=(3,)),
    configs.Workload("gathered_graph", B=1, H=2, D=128, F=9, T=1040, W=1, ref=0, block_size=80,
                     outlier_heads=(1,), seed=30),
], ids=lambda w: w.name)
def test_step_captured_in_a_cuda_graph_equals_eager(w):
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    plan = vd.attn_plan(w.F, w.T, w.W, w.ref, w.block_size)
    assert (plan.info.n_gathers > 0) == (w.name == "gathered_graph")
    ws = torch.empty(max(16, vd.key_stats_workspace_bytes(w.B, w.H, w.N, w.D)), dtype=torch.uint8,
                     device="cuda")
    st = vd.key_stats(q, k, w.scale, workspace=ws)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")

    def step():
        plan.rebuild()
        vd.key_stats(q, k, w.scale, workspace=ws, out=st)
        vd.attn_fwd(plan, q, k, v, st, w.scale, out=o, lse=lse, check=False)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm-up outside the capture (kernel attributes)
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want_o, want_l = o.clone(), lse.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert plan.status() == 0
        assert torch.equal(o.view(torch.int16), want_o.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), want_l.view(torch.int32))
    # new inputs written in place: the replay computes them, as the eager step does
    q2, k2, v2 = (t.cuda() for t in synth.make_qkv(w, seed=99))
    q.copy_(q2); k.copy_(k2); v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    got = o.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), o.view(torch.int16))
    assert not torch.equal(got.view(torch.int16), want_o.view(torch.int16))
