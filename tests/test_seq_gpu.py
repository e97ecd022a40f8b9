"""Parity of the sequence-split forward (kla_chunk_fwd_seq, through the C
ABI) with the oracle: the segments' zero-state and homogeneous runs, the
chained start states and the O_hom S correction together must give the
recurrence's o and final state within the bf16 bound (2e-2)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "eta")
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kla.load_library()
    yield
    assert kla.device_status() == 0


def rel_err(x, ref):
    x = x.detach().double().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run_seq(inp, segments, rule="kaczmarz", state=True):
    d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for n, v in inp.items()}
    o, hT = kla.chunk_fwd_seq(*[d[n] for n in NAMES], d["eps"], d["h0"],
                              C=64, segments=segments, rule=rule,
                              want_state=state)
    torch.cuda.synchronize()
    return o, hT


def oracle_fwd(inp):
    return oracle.kla_fwd(*[inp[n] for n in NAMES], inp["eps"], inp["h0"])


@pytest.mark.parametrize("segments", [2, 4, 8])
def test_segments_against_oracle(segments):
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=1024, H=2)
    o, hT = run_seq(inp, segments)
    o_ref, h_ref = oracle_fwd(inp)
    assert rel_err(o, o_ref) <= TOL and rel_err(hT, h_ref) <= TOL


def test_batches_initial_state_and_three_segments():
    """B = 2 with h0: segment 0 of each sequence starts from its own h0."""
    inp = gen.prefill_inputs(replace(gen.LAYER_1B, h0_std=0.3), B=2, T=768,
                             H=3)
    o, hT = run_seq(inp, 3)
    o_ref, h_ref = oracle_fwd(inp)
    assert rel_err(o, o_ref) <= TOL and rel_err(hT, h_ref) <= TOL


def test_learned_step_rule():
    """beta = eta given directly; the oracle runs it as KLA with eta' =
    b (||k||^2 + eps), the reduction the CPU pins check."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=512, H=2)
    b = np.random.default_rng(5).uniform(0.0, 0.5, inp["eta"].shape)
    inp["eta"] = torch.from_numpy(b.astype(np.float32))
    o, hT = run_seq(inp, 4, rule="given")
    k = inp["k"].double().numpy()
    ref_in = dict(inp)
    ref_in["eta"] = b.astype(np.float32).astype(np.float64) * (
        np.sum(k * k, -1) + inp["eps"])
    o_ref, h_ref = oracle_fwd(ref_in)
    assert rel_err(o, o_ref) <= TOL and rel_err(hT, h_ref) <= TOL


def test_one_segment_is_the_plain_forward():
    """One segment runs the fused tensor-core kernel on the whole sequence
    (the sequence path allocates nothing of its own), bit for bit."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=640, H=2)
    o1, h1 = run_seq(inp, 1)
    d = {n: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for n, v in inp.items()}
    o2, h2 = kla.chunk_fwd(*[d[n] for n in NAMES], d["eps"], d["h0"], C=64,
                           algo="tc_fused")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_without_final_state():
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=512, H=2)
    o, hT = run_seq(inp, 2, state=False)
    o_ref, _ = oracle_fwd(inp)
    assert hT is None and rel_err(o, o_ref) <= TOL


def test_long_context_with_outlier_keys_sampled_heads():
    """B1 T65536 H16 with 1% of keys at norm 10 and 1% at norm 0.05, split
    automatically; heads 2..3 followed by the oracle over every token."""
    inp = gen.prefill_inputs(gen.LONG_CTX)
    o, hT = run_seq(inp, 0)
    hs = slice(2, 4)
    sub = {n: (v[:, :, hs].contiguous() if n in NAMES else v)
           for n, v in inp.items()}
    o_ref, h_ref = oracle_fwd(sub)
    assert rel_err(o[:, :, hs], o_ref) <= TOL
    assert rel_err(hT[:, hs], h_ref) <= TOL


def test_131k_prefill_sampled_heads():
    """The 131072-token prefill split automatically; heads 11..12 followed
    by the oracle over every token."""
    inp = gen.prefill_inputs(gen.LONG_131K)
    o, hT = run_seq(inp, 0)
    hs = slice(11, 13)
    sub = {n: (v[:, :, hs].contiguous() if n in NAMES else v)
           for n, v in inp.items()}
    o_ref, h_ref = oracle_fwd(sub)
    assert rel_err(o[:, :, hs], o_ref) <= TOL
    assert rel_err(hT[:, hs], h_ref) <= TOL
