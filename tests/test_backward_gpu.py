"""Parity of the backward pass (kla_chunk_bwd, through the C ABI) with the
oracle's reverse mode of the fp64 recurrence.

Metric per gradient tensor: err = max|x - x_ref| / max|x_ref|.
Bounds: fp32 I/O <= 1e-4, bf16 I/O <= 2e-2 (as for the forward pass).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
NAMES = {"q_grad": "dq", "k_grad": "dk", "v_grad": "dv",
         "log_alpha_grad": "dlog_alpha", "eta_grad": "deta",
         "h0_grad": "dh0"}


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kla.load_library()
    yield
    assert kla.device_status() == 0


def rel_err(x, ref):
    x = x.detach().double().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def upstream(inp, seed, with_dhT=True):
    """Seeded dL/do (in the I/O dtype) and dL/dhT (fp32)."""
    rng = np.random.default_rng(seed)
    B, T, H, dv = inp["v"].shape
    dk = inp["k"].shape[-1]
    do = torch.from_numpy(rng.standard_normal((B, T, H, dv)).astype(
        np.float32)).to(inp["v"].dtype)
    dhT = (torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(
        np.float32)) if with_dhT else None)
    return do, dhT


def gpu_bwd(inp, do, dhT, C, rule="kaczmarz"):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in inp.items()}
    g = kla.chunk_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                      do.cuda(), None if dhT is None else dhT.cuda(),
                      eps=d["eps"], h0=d["h0"], C=C, rule=rule)
    torch.cuda.synchronize()
    return g


def check(inp, do, dhT, C, rule="kaczmarz"):
    g = gpu_bwd(inp, do, dhT, C, rule)
    ref = oracle.kla_bwd(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                         inp["eta"], inp["eps"], inp["h0"], do, dhT,
                         given=(rule == "given"))
    tol = TOL[inp["q"].dtype]
    errs = {}
    for name, key in NAMES.items():
        errs[name] = rel_err(g[name], ref[key])
        assert np.isfinite(errs[name]) and errs[name] <= tol, (name, errs)
    return errs


@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
@pytest.mark.parametrize("C,T", [(16, 64), (16, 50), (32, 64), (64, 64),
                                 (64, 130)])
def test_tiny_fp32(rule, C, T):
    inp = gen.prefill_inputs(gen.TINY, T=T)
    do, dhT = upstream(inp, 7 + T + C)
    check(inp, do, dhT, C, rule)


def test_tiny_fp32_with_initial_state_and_no_dhT():
    from dataclasses import replace
    w = replace(gen.TINY, h0_std=0.5)
    inp = gen.prefill_inputs(w, B=2, T=45, H=3)
    do, _ = upstream(inp, 11, with_dhT=False)
    check(inp, do, None, 16)


@pytest.mark.parametrize("dk,dv", [(32, 16), (16, 64), (64, 32)])
def test_fp32_head_dims(dk, dv):
    from dataclasses import replace
    w = replace(gen.TINY, dk=dk, dv=dv, h0_std=0.3)
    inp = gen.prefill_inputs(w, B=1, T=70, H=2)
    do, dhT = upstream(inp, dk + dv)
    check(inp, do, dhT, 32)


def test_fp32_many_heads_wide_state_slices():
    """B*H = 80 heads of dk = dv = 64: more (head, 32-column) slices than a
    GB300 has SMs, so the reverse state recurrence runs 64-column slices."""
    from dataclasses import replace
    w = replace(gen.TINY, dk=64, dv=64, h0_std=0.3)
    inp = gen.prefill_inputs(w, B=2, T=70, H=40)
    do, dhT = upstream(inp, 41)
    check(inp, do, dhT, 32)


@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
def test_bf16_d128(rule):
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=200, H=2)
    do, dhT = upstream(inp, 21)
    check(inp, do, dhT, 64, rule)


@pytest.mark.parametrize("dv", [64, 32])
def test_bf16_dk128_narrower_values(dv):
    """bf16, dk = 128, C = 64 with dv = 64 or 32: the checkpoints come from
    the CUDA-core forward and the per-chunk records from the backward's own
    pre-pass; dv = 64 runs the tensor-core recurrence, dv = 32 the
    CUDA-core one; both the tensor-core gradient kernel.  With h0 and a
    ragged last chunk."""
    from dataclasses import replace
    w = replace(gen.LAYER_1B, dv=dv)
    inp = gen.prefill_inputs(w, B=2, T=150, H=2)
    do, dhT = upstream(inp, 27)
    check(inp, do, dhT, 64)


def test_bf16_full_size_sampled_heads():
    """The 1B layer (B4 T4096 H16) on the GPU; heads (b=1, h=3..4) are
    followed by the oracle's reverse mode over all 4096 tokens."""
    inp = gen.prefill_inputs(gen.LAYER_1B)
    do, dhT = upstream(inp, 31)
    g = gpu_bwd(inp, do, dhT, 64)
    tok = np.s_[1:2, :, 3:5]        # [B, T, H, ...] tensors
    st = np.s_[1:2, 3:5]            # [B, H, dk, dv] tensors
    ref = oracle.kla_bwd(inp["q"][tok], inp["k"][tok], inp["v"][tok],
                         inp["log_alpha"][tok], inp["eta"][tok], inp["eps"],
                         inp["h0"][st], do[tok], dhT[st])
    for name, key in NAMES.items():
        got = g[name][st] if name == "h0_grad" else g[name][tok]
        e = rel_err(got, ref[key])
        assert np.isfinite(e) and e <= 2e-2, (name, e)


def test_zero_length_sequence_passes_state_gradient_through():
    inp = gen.prefill_inputs(gen.TINY, T=0)
    do, dhT = upstream(inp, 3)
    g = gpu_bwd(inp, do, dhT, 16)
    assert torch.equal(g["h0_grad"].cpu(), dhT)


def test_zero_keys_with_zero_eps():
    """beta := 0 where ||k||^2 + eps == 0: those tokens write nothing and
    get no eta gradient (as in the oracle)."""
    inp = gen.prefill_inputs(gen.TINY, T=40)
    inp["k"][:, 5:9] = 0.0
    inp["eps"] = 0.0
    do, dhT = upstream(inp, 5)
    check(inp, do, dhT, 16)
    g = gpu_bwd(inp, do, dhT, 16)
    assert torch.all(g["eta_grad"][:, 5:9] == 0)
