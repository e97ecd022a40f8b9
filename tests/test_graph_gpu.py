"""Decode steps captured in a CUDA graph (the library's launches are
capture-safe: no allocation, no synchronisation, no host read-back) give
exactly the state and outputs of the same steps launched one by one."""
import pytest
import torch

from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "eta")


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kla.load_library()
    yield
    assert kla.device_status() == 0


@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
def test_graph_replay_equals_eager_decode(rule):
    from dataclasses import replace
    w = replace(gen.DECODE, B=6, H=4)
    steps = 12
    d = gen.decode_inputs(w, steps=steps)
    toks = [[d[n][i].cuda() for n in NAMES] for i in range(steps)]
    S0 = d["S0"].cuda()

    S_e = S0.clone()
    o_e = torch.empty((w.B, w.H, w.dv), dtype=toks[0][0].dtype, device="cuda")
    outs_e = []
    for t in toks:
        kla.decode_step(*t, S_e, eps=d["eps"], o=o_e, rule=rule)
        outs_e.append(o_e.clone())

    S_g = S0.clone()
    o_g = torch.empty_like(o_e)
    outs_g = [torch.empty_like(o_e) for _ in range(steps)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):              # warm-up off the capture
        kla.decode_step(*toks[0], S0.clone(), eps=d["eps"], o=o_g, rule=rule)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i, t in enumerate(toks):
            kla.decode_step(*t, S_g, eps=d["eps"], o=o_g, rule=rule)
            outs_g[i].copy_(o_g)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(S_g, S_e)
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)
