"""The forward pass from host buffers (kla_chunk_fwd_host, through the C ABI):
the copies overlap the kernels segment by segment, and the result is
bit-identical to kla_chunk_fwd_ex on device copies of the same inputs (whose
parity with the oracle the other GPU tests establish); one case is also
checked against the oracle directly."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
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


def pinned(inp):
    return {n: (v.pin_memory() if isinstance(v, torch.Tensor) else v)
            for n, v in inp.items()}


def both_paths(inp, C, rule="kaczmarz", h0=True, state=True):
    h = pinned(inp)
    d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for n, v in inp.items()}
    o_d, hT_d = kla.chunk_fwd(*[d[n] for n in NAMES], d["eps"],
                              d["h0"] if h0 else None, C=C, rule=rule,
                              want_state=state)
    o_h, hT_h = kla.chunk_fwd_host(*[h[n] for n in NAMES], h["eps"],
                                   h["h0"] if h0 else None, C=C, rule=rule,
                                   want_state=state)
    torch.cuda.synchronize()
    return o_d.cpu(), (hT_d.cpu() if state else None), o_h, hT_h


@pytest.mark.parametrize("T", [1000, 20, 64])
@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
def test_bf16_d128_matches_device_path_bitwise(T, rule):
    """The tensor-core kernel per segment: 16 chunks in 8 segments with a
    ragged tail, one partial chunk, one whole chunk."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=T, H=4)
    o_d, hT_d, o_h, hT_h = both_paths(inp, 64, rule)
    assert torch.equal(o_d, o_h) and torch.equal(hT_d, hT_h)


def test_fp32_small_dims_match_device_path_bitwise():
    """The CUDA-core kernel per segment (fp32, d16, C16)."""
    inp = gen.prefill_inputs(replace(gen.TINY, h0_std=0.3), B=2, T=77, H=3)
    o_d, hT_d, o_h, hT_h = both_paths(inp, 16)
    assert torch.equal(o_d, o_h) and torch.equal(hT_d, hT_h)


def test_fp32_against_the_oracle():
    inp = gen.prefill_inputs(replace(gen.TINY, h0_std=0.3), B=2, T=150, H=2)
    h = pinned(inp)
    o, hT = kla.chunk_fwd_host(*[h[n] for n in NAMES], h["eps"], h["h0"],
                               C=16)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.kla_fwd(*[inp[n] for n in NAMES], inp["eps"],
                                  inp["h0"])
    err = lambda x, r: float(np.max(np.abs(x.double().numpy() - r)) /
                             np.max(np.abs(r)))
    assert err(o, o_ref) <= 1e-4 and err(hT, h_ref) <= 1e-4


def test_no_initial_state_and_no_final_state():
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=300, H=2)
    o_d, _, o_h, hT_h = both_paths(inp, 64, h0=False, state=False)
    assert hT_h is None and torch.equal(o_d, o_h)


def test_zero_length_sequence():
    inp = gen.prefill_inputs(replace(gen.TINY, h0_std=0.5), B=2, T=0, H=3)
    h = pinned(inp)
    _, hT = kla.chunk_fwd_host(*[h[n] for n in NAMES], h["eps"], h["h0"],
                               C=16)
    _, hz = kla.chunk_fwd_host(*[h[n] for n in NAMES], h["eps"], None, C=16)
    torch.cuda.synchronize()
    assert torch.equal(hT, inp["h0"]) and torch.count_nonzero(hz) == 0


def test_repeated_calls_share_a_workspace():
    """Back-to-back calls on one stream with one workspace (the library's
    copy streams and events are reused): each call's result stands."""
    a = pinned(gen.prefill_inputs(gen.LAYER_1B, B=2, T=700, H=2))
    b = pinned(gen.prefill_inputs(gen.LAYER_1B, seed=77, B=2, T=700, H=2))
    ws = torch.empty(kla.chunk_fwd_host_workspace_size(2, 700, 2, 128, 128,
                                                       64, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    outs = [kla.chunk_fwd_host(*[x[n] for n in NAMES], x["eps"], x["h0"],
                               C=64, workspace=ws) for x in (a, b, a)]
    torch.cuda.synchronize()
    ref = [kla.chunk_fwd(*[x[n].cuda() for n in NAMES], x["eps"],
                         x["h0"].cuda(), C=64) for x in (a, b)]
    torch.cuda.synchronize()
    for (o, hT), (o_r, h_r) in zip(outs, ref + ref[:1]):
        assert torch.equal(o, o_r.cpu()) and torch.equal(hT, h_r.cpu())


def test_full_size_matches_device_path_bitwise():
    """The 1B layer (B4 T4096 H16 d128) through host buffers."""
    inp = gen.prefill_inputs(gen.LAYER_1B)
    o_d, hT_d, o_h, hT_h = both_paths(inp, 64)
    assert torch.equal(o_d, o_h) and torch.equal(hT_d, hT_h)
