"""kla_chunk_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (no allocator of their own, or a fixed memory budget), with
its scratch in a fixed 32 MiB array inside the library.

This file is named so that pytest collects it last: its GPU test checks the
entry point against kla_chunk_bwd (caller-provided workspace) on three calls
in a row -- the largest problem of its shape that fits the array, a small
one, then the large one again with new inputs, so that the third call finds
the first two calls' contents all over the array; it must pass both alone in
a fresh process and after every other test.
"""
import ctypes
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

GRADS = ("q_grad", "k_grad", "v_grad", "log_alpha_grad", "eta_grad",
         "h0_grad")
ORACLE_KEYS = {"q_grad": "dq", "k_grad": "dk", "v_grad": "dv",
               "log_alpha_grad": "dlog_alpha", "eta_grad": "deta",
               "h0_grad": "dh0"}
LIMIT = 32 << 20
# per (batch, head, chunk) with dk = dv = 128, C = 64: two fp32 128 x 128
# states, the backward's 17,152-byte record and the forward pre-pass's
# 16,640-byte one with its 4-byte ready flag, plus 528 bytes of the
# pre-pass's work counters in all; B1 H4 T3200 is 200 chunks, the most of
# whole chunks that fit (203 would; 204, at T = 3201, do not)
PER_CHUNK = 2 * 128 * 128 * 4 + 17152 + 16640 + 4
FIXED = 528
FULL = dict(B=1, T=3200, H=4)


def _call(lib, T, q=0x10000):
    Q = None if q is None else ctypes.c_void_p(q)
    # distinct fake buffers far apart, so that no overlap check fires
    b = [ctypes.c_void_p(0x10000 + (i << 32)) for i in range(12)]
    return lib.kla_chunk_bwd_noalloc(Q, b[1], b[2], b[3], b[4], 1e-6, None,
                                     b[5], None, b[6], b[7], b[8], b[9],
                                     b[10], None, 1, T, 4, 128, 128, 64, 1, 0,
                                     None)


def test_size_limit_is_checked_after_the_arguments():
    """Host-side only (nothing is launched on any of these paths): the
    workspace of B1 T3200 H4 d128 C64 is 200 chunk records and fits in the
    32 MiB; one more token (four more chunks) does not and is refused with
    KLA_ERR_UNSUPPORTED_SHAPE; a null input is reported as
    KLA_ERR_INVALID_ARG even when the problem is too large."""
    lib = kla.load_library()
    assert kla.chunk_bwd_workspace_size(FULL["B"], FULL["T"], FULL["H"],
                                        128, 128, 64) == \
        200 * PER_CHUNK + FIXED
    assert 200 * PER_CHUNK + FIXED <= LIMIT < 204 * PER_CHUNK + FIXED
    assert kla.chunk_bwd_workspace_size(1, 3201, 4, 128, 128, 64) > LIMIT
    assert _call(lib, 3201) == -2          # KLA_ERR_UNSUPPORTED_SHAPE
    assert _call(lib, 3201, q=None) == -1  # KLA_ERR_INVALID_ARG first
    assert _call(lib, 1 << 20) == -2


def _case(w, seed, **sizes):
    inp = gen.prefill_inputs(w, **sizes)
    rng = np.random.default_rng(seed)
    B, T, H, dv = inp["v"].shape
    dk = inp["k"].shape[-1]
    do = torch.from_numpy(rng.standard_normal((B, T, H, dv)).astype(
        np.float32)).to(inp["v"].dtype)
    dhT = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(
        np.float32))
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in inp.items()}
    return inp, d, do, dhT


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_three_calls():
    """Three calls in a row: the largest 1B-layer-shaped problem that fits
    the array, a small fp32 one, then the large one again on new inputs.  Each result equals the one
    kla_chunk_bwd gives with a caller-allocated workspace up to the order of
    the kernels' atomic sums; the small one and the last large one are also
    held to the oracle's reverse mode at the fp32 / bf16 bounds."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    cases = [(gen.LAYER_1B, 61, FULL, False),
             (replace(gen.TINY, h0_std=0.5), 62, dict(B=2, T=100, H=3), True),
             (gen.LAYER_1B, 63, FULL, True)]
    for w, seed, sizes, vs_oracle in cases:
        inp, d, do, dhT = _case(w, seed, **sizes)
        args = (d["q"], d["k"], d["v"], d["log_alpha"], d["eta"], do.cuda(),
                dhT.cuda())
        kw = dict(eps=d["eps"], h0=d["h0"], C=w.C)
        ref = kla.chunk_bwd(*args, **kw)
        got = kla.chunk_bwd_noalloc(*args, **kw)
        torch.cuda.synchronize()
        for name in GRADS:
            x, r = got[name], ref[name]
            assert x.dtype == r.dtype
            xd, rd = x.double(), r.double()
            scale = float(rd.abs().max().clamp_min(1e-30))
            # one bf16 rounding step of the element for bf16 outputs, plus
            # fp32 summation-order noise relative to the tensor's maximum
            ulp = 2.0 ** -7 if x.dtype == torch.bfloat16 else 0.0
            bound = ulp * rd.abs() + 1e-5 * scale
            assert bool(((xd - rd).abs() <= bound).all()), (w.name, name)
        if vs_oracle:
            g = oracle.kla_bwd(*[inp[n] for n in ("q", "k", "v", "log_alpha",
                                                  "eta")],
                               inp["eps"], inp["h0"], do, dhT)
            tol = 1e-4 if d["q"].dtype == torch.float32 else 2e-2
            for name in GRADS:
                ref_o = g[ORACLE_KEYS[name]]
                x = got[name].double().cpu().numpy()
                err = float(np.max(np.abs(x - ref_o)) /
                            max(np.max(np.abs(ref_o)), 1e-30))
                assert np.isfinite(err) and err <= tol, (w.name, name, err)
    assert kla.device_status() == 0
