"""The compute entry points enqueue only kernels and asynchronous memsets on
the caller's stream (no allocation, no synchronisation), so a serving or
training loop can capture them in a CUDA graph.  Captured-and-replayed results
equal the eager results bit for bit, also after the inputs are overwritten in
place between replays."""

import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth

pytestmark = pytest.mark.gpu
V1 = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up launch outside the graph (first-use host work)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_v2_decode_graph_replay():
    t = synth.decode_inputs(4, 2048, 32, 8, 128, 512, seed=9100, device="cuda", seqlens=[2048, 1000, 77, 1])
    need = bd.diffattn_v2_decode_workspace_size(4, 32, 8, 128, 2048)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    out = torch.empty((4, 32, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"], x=t["x"],
                              w_lambda=t["w_lambda"], out=out, workspace=ws)

    g = _capture(step)
    for seed in (9101, 9102):
        u = synth.decode_inputs(4, 2048, 32, 8, 128, 512, seed=seed, device="cuda")
        t["q"].copy_(u["q"])
        t["x"].copy_(u["x"])
        g.replay()
        torch.cuda.synchronize()
        eager = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"], x=t["x"],
                                      w_lambda=t["w_lambda"])
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


def test_v1_fwd_graph_replay():
    """The V1 forward's work counter is reset by a memset node inside the graph."""
    t = synth.v1_inputs(2, 640, 3, 128, 256, "bf16", seed=9200, device="cuda")
    li = bd.diffattn_lambda_init(2)
    need = bd.load().diffattn_v1_fwd_workspace_size(2, 640, 3, 128, 256, bd.DA_BF16)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, 640, 3, 256), dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: bd.diffattn_v1_fwd(*(t[n] for n in V1), li, out=out, workspace=ws))
    for rep in range(3):  # the counter must start from zero on every replay
        g.replay()
        torch.cuda.synchronize()
        eager = bd.diffattn_v1_fwd(*(t[n] for n in V1), li)
        torch.cuda.synchronize()
        assert torch.equal(out, eager), rep


def test_v2_fwd_graph_replay():
    t = synth.v2_inputs(1, 700, 4, 2, 128, 256, seed=9300, device="cuda")
    need = bd.load().diffattn_v2_fwd_workspace_size(1, 700, 4, 0)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 700, 4, 128), dtype=torch.bfloat16, device="cuda")
    g = _capture(lambda: bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], out=out,
                                            workspace=ws))
    t["q"].mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    eager = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
