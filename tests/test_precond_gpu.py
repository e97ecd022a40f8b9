"""Parity of the diagonal-preconditioned variant (kla_precond_keys,
kla_chunk_fwd_kw, kla_decode_step_kw; through the C ABI) with the oracle's
preconditioned recurrence.

Metric per tensor: err = max|x - x_ref| / max|x_ref|; fp32 I/O <= 1e-4,
bf16 I/O <= 2e-2.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
X, DELTA = 1.5, 1e-6


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kla.load_library()
    yield
    assert kla.device_status() == 0


def rel_err(x, ref):
    x = x.detach().double().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def aniso(inp, seed):
    """Per-dimension key scales, so that the preconditioner matters."""
    rng = np.random.default_rng(seed)
    dk = inp["k"].shape[-1]
    s = torch.from_numpy(rng.uniform(0.3, 3.0, dk).astype(np.float32))
    inp = dict(inp)
    inp["k"] = (inp["k"].float() * s).to(inp["k"].dtype)
    return inp


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
            for k, v in inp.items()}


@pytest.mark.parametrize("w,sizes", [
    (gen.TINY, dict(T=50)),
    (gen.TINY, dict(T=0)),
    (replace(gen.TINY, dk=32, dv=32), dict(T=777)),
    (replace(gen.TINY, dk=64), dict(B=1, T=1029, H=3)),
    (gen.LAYER_1B, dict(B=2, T=1, H=2)),
    (gen.LAYER_1B, dict(B=2, T=64, H=3)),
    (gen.LAYER_1B, dict(B=2, T=65, H=2)),
    (gen.LAYER_1B, dict(B=2, T=300, H=2)),
    (gen.LAYER_1B, dict(B=1, T=4096, H=2)),
    (gen.LAYER_1B, dict(B=1, T=4100, H=2)),
    (replace(gen.LAYER_1B, dtype="f32"), dict(B=1, T=2048, H=2)),
    (replace(gen.LAYER_1B, dtype="f32"), dict(B=1, T=2100, H=3)),
])
def test_write_keys_and_second_moments(w, sizes):
    """dk = 128 takes the chunked form: one launch from A0 for a single
    chunk (T = 1, 64), else sums, scan and weighting over 64-token chunks
    (T = 65: a one-token last chunk; 300, 2100: ragged; 4100: 65 chunks,
    two batches of the scan's loads); other dk the cluster kernel."""
    inp = aniso(gen.prefill_inputs(w, **sizes), 1)
    B, T, H, dk = inp["k"].shape
    A0 = torch.from_numpy(np.random.default_rng(2).uniform(
        0, 5, (B, H, dk)).astype(np.float32))
    d = dev(inp)
    kw, AT = kla.precond_keys(d["k"], A0.cuda(), x=X, delta=DELTA)
    torch.cuda.synchronize()
    _, _, A_ref, kw_ref = oracle.pkla_fwd(inp["q"], inp["k"], inp["v"],
                                          inp["log_alpha"], inp["eta"],
                                          inp["eps"], None, A0=A0, x=X,
                                          delta=DELTA)
    tol = TOL[inp["k"].dtype]
    if T == 0:
        assert torch.equal(AT.cpu(), A0)
        return
    assert rel_err(kw, kw_ref) <= tol
    assert rel_err(AT, A_ref) <= 1e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_write_keys_misaligned_take_the_cluster_kernel(dtype):
    """dk = 128 keys that are not 16-byte aligned (a view one element into
    its buffer) take the cluster kernel; same bounds against the oracle."""
    w = gen.LAYER_1B if dtype == torch.bfloat16 else \
        replace(gen.LAYER_1B, dtype="f32")
    inp = aniso(gen.prefill_inputs(w, B=1, T=200, H=2), 7)
    B, T, H, dk = inp["k"].shape
    buf = torch.empty(inp["k"].numel() + 1, dtype=dtype, device="cuda")
    k = buf[1:].view(B, T, H, dk)
    k.copy_(inp["k"].cuda())
    assert k.data_ptr() % 16 != 0
    kw, AT = kla.precond_keys(k, None, x=X, delta=DELTA)
    torch.cuda.synchronize()
    _, _, A_ref, kw_ref = oracle.pkla_fwd(inp["q"], inp["k"], inp["v"],
                                          inp["log_alpha"], inp["eta"],
                                          inp["eps"], None, x=X, delta=DELTA)
    assert rel_err(kw, kw_ref) <= TOL[dtype]
    assert rel_err(AT, A_ref) <= 1e-5


def test_write_keys_plain_entry_point_equals_workspace_form():
    """kla_precond_keys (the library's stream-ordered scratch) and
    kla_precond_keys_ex with a caller workspace run the same kernels: the
    same bits."""
    import ctypes
    inp = aniso(gen.prefill_inputs(gen.LAYER_1B, B=2, T=700, H=3), 8)
    k = inp["k"].cuda()
    B, T, H, dk = k.shape
    A0 = torch.rand(B, H, dk, device="cuda") * 4
    kw1, AT1 = kla.precond_keys(k, A0, x=X, delta=DELTA)
    kw2, AT2 = torch.empty_like(k), torch.empty_like(A0)
    st = kla.load_library().kla_precond_keys(
        ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(A0.data_ptr()),
        ctypes.c_void_p(kw2.data_ptr()), ctypes.c_void_p(AT2.data_ptr()),
        B, T, H, dk, X, DELTA, kla.DTYPES[k.dtype],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(kw1, kw2) and torch.equal(AT1, AT2)


@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
@pytest.mark.parametrize("C,T", [(16, 64), (16, 50), (64, 130)])
def test_forward_fp32(rule, C, T):
    w = replace(gen.TINY, h0_std=0.3)
    inp = aniso(gen.prefill_inputs(w, B=2, T=T, H=2), 3)
    d = dev(inp)
    kw, _ = kla.precond_keys(d["k"], x=X, delta=DELTA)
    o, hT = kla.chunk_fwd_kw(d["q"], d["k"], kw, d["v"], d["log_alpha"],
                             d["eta"], d["eps"], d["h0"], C=C, rule=rule)
    torch.cuda.synchronize()
    o_ref, h_ref, _, _ = oracle.pkla_fwd(inp["q"], inp["k"], inp["v"],
                                         inp["log_alpha"], inp["eta"],
                                         inp["eps"], inp["h0"], x=X,
                                         delta=DELTA, given=(rule == "given"))
    assert rel_err(o, o_ref) <= 1e-4 and rel_err(hT, h_ref) <= 1e-4


@pytest.mark.parametrize("algo", ["tc", "tc_fused"])
@pytest.mark.parametrize("rule", ["kaczmarz", "given"])
@pytest.mark.parametrize("T", [50, 128, 400])
def test_forward_bf16_d128(rule, T, algo):
    """bf16, dk = dv = 128, C = 64: the write-key modes of the two-kernel
    path and of the fused tensor-core kernel (one chunk, whole chunks, a
    ragged tail)."""
    inp = aniso(gen.prefill_inputs(gen.LAYER_1B, B=1, T=T, H=2), 4)
    d = dev(inp)
    kw, _ = kla.precond_keys(d["k"], x=X, delta=DELTA)
    o, hT = kla.chunk_fwd_kw(d["q"], d["k"], kw, d["v"], d["log_alpha"],
                             d["eta"], d["eps"], d["h0"], C=64, rule=rule,
                             algo=algo)
    torch.cuda.synchronize()
    o_ref, h_ref, _, _ = oracle.pkla_fwd(inp["q"], inp["k"], inp["v"],
                                         inp["log_alpha"], inp["eta"],
                                         inp["eps"], inp["h0"], x=X,
                                         delta=DELTA, given=(rule == "given"))
    assert rel_err(o, o_ref) <= 2e-2 and rel_err(hT, h_ref) <= 2e-2


def test_prefill_then_decode_handoff():
    """Prefill of 100 tokens (write keys + two-key forward), then 20 decode
    steps (write key of one token + two-key decode step), the second moments
    and the state carried across; equals the oracle over all 120 tokens."""
    inp = aniso(gen.prefill_inputs(gen.LAYER_1B, B=2, T=120, H=2), 5)
    o_ref, h_ref, A_ref, _ = oracle.pkla_fwd(
        inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["eta"],
        inp["eps"], inp["h0"], x=X, delta=DELTA)
    d = dev(inp)
    sl = slice(0, 100)
    cut = {n: d[n][:, sl].contiguous()
           for n in ("q", "k", "v", "log_alpha", "eta")}
    kw, A = kla.precond_keys(cut["k"], x=X, delta=DELTA)
    o, S = kla.chunk_fwd_kw(cut["q"], cut["k"], kw, cut["v"],
                            cut["log_alpha"], cut["eta"], d["eps"], d["h0"],
                            C=64)
    outs = [o]
    for t in range(100, 120):
        tok = {n: d[n][:, t].contiguous()
               for n in ("q", "k", "v", "log_alpha", "eta")}
        kwt, A = kla.precond_keys(tok["k"][:, None].contiguous(), A, x=X,
                                  delta=DELTA, AT=A)
        outs.append(kla.decode_step_kw(
            tok["q"], tok["k"], kwt[:, 0].contiguous(), tok["v"],
            tok["log_alpha"], tok["eta"], S, eps=d["eps"])[:, None])
    torch.cuda.synchronize()
    assert rel_err(torch.cat(outs, 1), o_ref) <= 2e-2
    assert rel_err(S, h_ref) <= 2e-2
    assert rel_err(A, A_ref) <= 1e-5


@pytest.mark.parametrize("algo", ["tc", "tc_fused"])
def test_write_keys_equal_to_keys_give_the_plain_forward(algo):
    """With k_write = k the write-key mode of each tensor-core path computes
    exactly what its plain mode does (same operands, same order): o and the
    state are bit-identical."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=300, H=3)
    d = dev(inp)
    o1, h1 = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                           d["eps"], d["h0"], C=64, algo=algo)
    o2, h2 = kla.chunk_fwd_kw(d["q"], d["k"], d["k"], d["v"],
                              d["log_alpha"], d["eta"], d["eps"], d["h0"],
                              C=64, algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_forward_full_size_sampled_heads():
    """The 1B layer (B4 T4096 H16) through write keys and the two-key
    forward on the GPU; heads (b=2, h=7..8) follow the oracle over all 4096
    tokens."""
    inp = aniso(gen.prefill_inputs(gen.LAYER_1B), 6)
    d = dev(inp)
    kw, _ = kla.precond_keys(d["k"], x=X, delta=DELTA)
    o, hT = kla.chunk_fwd_kw(d["q"], d["k"], kw, d["v"], d["log_alpha"],
                             d["eta"], d["eps"], d["h0"], C=64)
    torch.cuda.synchronize()
    tok = np.s_[2:3, :, 7:9]
    st = np.s_[2:3, 7:9]
    o_ref, h_ref, _, _ = oracle.pkla_fwd(
        inp["q"][tok], inp["k"][tok], inp["v"][tok], inp["log_alpha"][tok],
        inp["eta"][tok], inp["eps"], inp["h0"][st], x=X, delta=DELTA)
    assert rel_err(o[tok], o_ref) <= 2e-2
    assert rel_err(hT[st], h_ref) <= 2e-2

