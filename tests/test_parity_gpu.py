"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Metric (per output tensor): err = max|x - x_ref| / max|x_ref|.
Bounds: fp32 I/O <= 1e-4, bf16 I/O <= 2e-2, for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_delta_gb300 import inputs as gen
from linear_attention_delta_gb300 import kla

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    kla.load_library()
    yield
    assert kla.device_status() == 0


def rel_err(x, ref):
    x = x.detach().double().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def to_dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
            for k, v in d.items()}


def run_fwd(inp, algo="auto", C=None):
    d = to_dev(inp)
    o, hT = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                          d["eps"], d["h0"], C=C or inp["C"], algo=algo)
    torch.cuda.synchronize()
    return o, hT


def oracle_fwd(inp):
    return oracle.kla_fwd(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                          inp["eta"], inp["eps"], inp["h0"])


def check_fwd(inp, algo="auto", C=None):
    o, hT = run_fwd(inp, algo, C)
    o_ref, h_ref = oracle_fwd(inp)
    tol = TOL[inp["q"].dtype]
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    assert np.isfinite(eo) and eo <= tol, f"o err {eo:.3e} > {tol}"
    assert np.isfinite(eh) and eh <= tol, f"hT err {eh:.3e} > {tol}"
    return eo, eh


# ---------------------------------------------------------------- tiny fp32

@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_tiny_fp32(algo):
    check_fwd(gen.prefill_inputs(gen.TINY), algo)


def test_tiny_unrelaxed_projection_through_gpu():
    """eta=1, eps=0, alpha=1: with q := k every output equals its value
    (S_t^T k_t = v_t, the projection property) through the CUDA path."""
    inp = gen.prefill_inputs(gen.TINY_UNRELAXED)
    inp["q"] = inp["k"].clone()
    o, _ = run_fwd(inp)
    assert rel_err(o, inp["v"].double().numpy()) <= 1e-4
    check_fwd(inp)


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 17, 64, 100])
def test_fp32_chunk_sizes_and_ragged_tails(C, T):
    inp = gen.prefill_inputs(gen.TINY, T=T, B=2, H=3)
    check_fwd(inp, "simt", C)


@pytest.mark.parametrize("dk,dv", [(16, 32), (32, 16), (64, 64), (128, 16),
                                   (32, 128)])
def test_fp32_head_dims(dk, dv):
    from dataclasses import replace
    w = replace(gen.TINY, dk=dk, dv=dv)
    check_fwd(gen.prefill_inputs(w, T=40, B=1, H=2), "simt", 16)


# ---------------------------------------------------------------- bf16 d=128

SMALL_BF16 = [
    (gen.LAYER_340M, dict(B=2, T=200, H=3)),
    (gen.LAYER_1B, dict(B=1, T=257, H=4)),
    (gen.LONG_CTX, dict(B=1, T=1000, H=2)),
]


@pytest.mark.parametrize("w,sizes", SMALL_BF16,
                         ids=[w.name for w, _ in SMALL_BF16])
@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_bf16_reduced_sizes(w, sizes, algo):
    check_fwd(gen.prefill_inputs(w, **sizes), algo)


def test_bf16_chunk_size_invariance():
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=192, H=2)
    outs = [run_fwd(inp, "simt", C) for C in (16, 32, 64)]
    o_ref, h_ref = oracle_fwd(inp)
    for o, hT in outs:
        assert rel_err(o, o_ref) <= 2e-2 and rel_err(hT, h_ref) <= 2e-2
    assert rel_err(outs[0][1], outs[2][1].double().cpu().numpy()) <= 1e-3


def test_zero_length_sequence_copies_state():
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=0, H=2)
    o, hT = run_fwd(inp)
    assert o.numel() == 0
    assert torch.equal(hT.cpu(), inp["h0"])


def test_hT_may_alias_h0():
    inp = gen.prefill_inputs(gen.LAYER_1B, B=1, T=130, H=2)
    d = to_dev(inp)
    h = d["h0"].clone()
    kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"], d["eps"],
                  h, C=64, hT=h)
    torch.cuda.synchronize()
    _, h_ref = oracle_fwd(inp)
    assert rel_err(h, h_ref) <= 2e-2


def test_zero_keys_with_zero_eps():
    inp = gen.prefill_inputs(gen.TINY, B=1, T=48, H=2)
    inp["k"][:, 5] = 0.0
    inp["k"][:, 30:33] = 0.0
    inp["eps"] = 0.0
    check_fwd(inp, "simt")


@pytest.mark.parametrize("algo", ["tc", "tc_fused"])
def test_tensor_core_zero_keys_with_zero_eps(algo):
    """k = 0 with eps = 0 makes beta's denominator exactly 0; beta := 0 (no
    write), as in the oracle.  Through both tensor-core paths, with zero
    keys on the first and the last row of a chunk, inside a chunk, on a run
    of rows and on the last token of a ragged tail."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=200, H=2)
    for t in (0, 5, 63, 64, 100, 101, 102, 127, 199):
        inp["k"][:, t] = 0.0
    inp["k"][1, 130:140, 1] = 0.0
    inp["eps"] = 0.0
    check_fwd(inp, algo)


@pytest.mark.parametrize("algo", ["tc", "tc_fused"])
def test_tensor_core_unrelaxed_projection(algo):
    """eta = 1, eps = 0, alpha = 1 (every write an exact projection,
    S_t^T k_t = v_t): with q := k both bf16 tensor-core paths return each
    token's value, within the bf16 bound, over 3 chunks and a ragged tail."""
    from dataclasses import replace
    w = replace(gen.LAYER_1B, unrelaxed=True, eps=0.0, h0_std=0.0)
    inp = gen.prefill_inputs(w, B=1, T=200, H=2)
    assert float(inp["eps"]) == 0.0 and float(inp["eta"].min()) == 1.0
    assert float(inp["log_alpha"].abs().max()) == 0.0
    inp["q"] = inp["k"].clone()
    o, _ = run_fwd(inp, algo)
    assert rel_err(o, inp["v"].double().numpy()) <= 2e-2
    check_fwd(inp, algo)


def test_plain_c_entry_points_through_ctypes():
    """The two entry points of the boundary under their plain names,
    kla_chunk_fwd and kla_decode_step, called through ctypes on device
    buffers (no binding helper in between) and held to the oracle."""
    import ctypes
    lib = kla.load_library()
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=200, H=2)
    d = to_dev(inp)
    B, T, H, dk = inp["k"].shape
    dv = inp["v"].shape[-1]
    o = torch.empty_like(d["v"])
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    st = lib.kla_chunk_fwd(P(d["q"]), P(d["k"]), P(d["v"]),
                           P(d["log_alpha"]), P(d["eta"]),
                           ctypes.c_float(inp["eps"]), P(d["h0"]), P(o),
                           P(hT), B, T, H, dk, dv, 64, 1, stream)
    assert st == 0
    torch.cuda.synchronize()
    o_ref, h_ref = oracle_fwd(inp)
    assert rel_err(o, o_ref) <= 2e-2 and rel_err(hT, h_ref) <= 2e-2
    # three decode steps continuing from hT, plain kla_decode_step
    from dataclasses import replace
    dw = replace(gen.DECODE, B=B, H=H)
    dec = gen.decode_inputs(dw, steps=3)
    S = hT.clone()
    S_ref = h_ref
    for t in range(3):
        args = [dec[n][t] for n in ("q", "k", "v", "log_alpha", "eta")]
        dargs = [a.cuda() for a in args]
        od = torch.empty_like(dargs[2])
        st = lib.kla_decode_step(*[P(a) for a in dargs],
                                 ctypes.c_float(dec["eps"]), P(S), P(od),
                                 B, H, dk, dv, 1, stream)
        assert st == 0
        od_ref, S_ref = oracle.kla_decode_step(*args, dec["eps"], S_ref)
        torch.cuda.synchronize()
        assert rel_err(od, od_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("w", [gen.LAYER_340M, gen.LAYER_1B, gen.LONG_CTX],
                         ids=lambda w: w.name)
def test_full_size_against_oracle(w):
    """The workloads at their full sizes, every element compared (the
    default path: the two-kernel tensor-core forward)."""
    check_fwd(gen.prefill_inputs(w))


def test_full_size_fused_kernel_against_oracle():
    """The fused tensor-core kernel on the full 1B layer, every element."""
    check_fwd(gen.prefill_inputs(gen.LAYER_1B), "tc_fused")


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(16, 16), (128, 128), (64, 32),
                                   (32, 128)])
def test_decode_steps(dtype, dk, dv):
    from dataclasses import replace
    w = replace(gen.DECODE, dtype=dtype, dk=dk, dv=dv, B=5, H=3)
    d = gen.decode_inputs(w, steps=6)
    S = d["S0"].cuda()
    S_ref = d["S0"].double().numpy()
    tol = TOL[d["q"].dtype]
    for t in range(6):
        args = [d[n][t] for n in ("q", "k", "v", "log_alpha", "eta")]
        o = kla.decode_step(*[a.cuda() for a in args], S, eps=d["eps"])
        o_ref, S_ref = oracle.kla_decode_step(*args, d["eps"], S_ref)
        assert rel_err(o, o_ref) <= tol
    torch.cuda.synchronize()
    assert rel_err(S, S_ref) <= 1e-4


def test_decode_full_size_1000_steps():
    """The decode workload as specified: 256 sequences x 16 heads, 1000
    consecutive steps on the GPU (each step reads and writes the whole
    state).  The first 32 sequences (all 16 heads) are followed by the
    oracle through all 1000 steps -- as one fp64 recurrence over 1000 tokens
    per sequence, which the oracle pins show equals 1000 decode steps -- and
    o is compared at every step, the state after the last."""
    w = gen.DECODE
    steps, ns = w.T, 32
    d = gen.decode_inputs(w, steps=steps)
    dd = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
          for k, v in d.items()}
    S = dd["S0"].clone()
    outs = torch.empty((steps, ns) + tuple(d["v"].shape[2:]),
                       dtype=d["v"].dtype, device="cuda")
    for t in range(steps):
        o = kla.decode_step(dd["q"][t], dd["k"][t], dd["v"][t],
                            dd["log_alpha"][t], dd["eta"][t], S, eps=d["eps"])
        outs[t] = o[:ns]
    torch.cuda.synchronize()
    # [steps, N, H, d] -> [N, steps, H, d]: sequence n's tokens in order
    seq = {n: d[n][:, :ns].transpose(0, 1).contiguous()
           for n in ("q", "k", "v", "log_alpha", "eta")}
    o_ref, S_ref = oracle.kla_fwd(seq["q"], seq["k"], seq["v"],
                                  seq["log_alpha"], seq["eta"], d["eps"],
                                  d["S0"][:ns])
    o_gpu = outs.transpose(0, 1).double().cpu().numpy()
    per_step = [rel_err(o_gpu[:, t], o_ref[:, t]) for t in range(steps)]
    assert max(per_step) <= 2e-2, (int(np.argmax(per_step)), max(per_step))
    assert rel_err(S[:ns], S_ref) <= 1e-4


def test_prefill_then_decode_handoff():
    """A forward pass over the first 100 tokens followed by decode steps for
    the next 20 equals one recurrence over all 120 tokens."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=120, H=2)
    o_ref, h_ref = oracle_fwd(inp)
    d = to_dev(inp)
    sl = slice(0, 100)
    o, S = kla.chunk_fwd(d["q"][:, sl].contiguous(), d["k"][:, sl].contiguous(),
                         d["v"][:, sl].contiguous(),
                         d["log_alpha"][:, sl].contiguous(),
                         d["eta"][:, sl].contiguous(), d["eps"], d["h0"],
                         C=64)
    outs = [o]
    for t in range(100, 120):
        outs.append(kla.decode_step(
            d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
            d["v"][:, t].contiguous(), d["log_alpha"][:, t].contiguous(),
            d["eta"][:, t].contiguous(), S, eps=d["eps"])[:, None])
    torch.cuda.synchronize()
    assert rel_err(torch.cat(outs, 1), o_ref) <= 2e-2
    assert rel_err(S, h_ref) <= 2e-2


# ---------------------------------------------------------------- the pages' points

def test_long_prefill_131k_sampled_heads():
    """The 131072-token prefill (one sequence, 16 heads) on the GPU; four
    heads are followed by the oracle over every token (o and the final state
    of those heads compared element by element)."""
    inp = gen.prefill_inputs(gen.LONG_131K)
    o, hT = run_fwd(inp)
    hs = slice(5, 9)
    sub = {k: (v[:, :, hs].contiguous()
               if k in ("q", "k", "v", "log_alpha", "eta") else v)
           for k, v in inp.items()}
    assert sub["h0"] is None
    o_ref, h_ref = oracle_fwd(sub)
    assert rel_err(o[:, :, hs], o_ref) <= 2e-2
    assert rel_err(hT[:, hs], h_ref) <= 2e-2


def test_decode_after_32k_prefill():
    """Four sequences prefilled over 32768 tokens, then 40 decode steps from
    the prefill's final state; sequence 0 (all 16 heads) is followed by the
    oracle through the prefill and every decode step."""
    w = gen.HANDOFF_32K
    inp = gen.prefill_inputs(w)
    _, S = run_fwd(inp)
    sub = {k: (v[:1].contiguous() if isinstance(v, torch.Tensor) else v)
           for k, v in inp.items()}
    _, S_ref = oracle_fwd(sub)
    steps = 40
    d = gen.decode_inputs(w, steps=steps, seed=gen.SEEDS[w.name] + 100)
    dd = to_dev(d)
    worst = 0.0
    for t in range(steps):
        o = kla.decode_step(dd["q"][t], dd["k"][t], dd["v"][t],
                            dd["log_alpha"][t], dd["eta"][t], S,
                            eps=d["eps"])
        o_ref, S_ref = oracle.kla_decode_step(
            d["q"][t, :1], d["k"][t, :1], d["v"][t, :1],
            d["log_alpha"][t, :1], d["eta"][t, :1], d["eps"], S_ref)
        worst = max(worst, rel_err(o[:1], o_ref))
    torch.cuda.synchronize()
    assert worst <= 2e-2
    assert rel_err(S[:1], S_ref) <= 2e-2


# ---------------------------------------------------------------- kernel paths

@pytest.mark.parametrize("T", [64, 65, 128, 200, 1000])
def test_tensor_core_path_against_oracle(T):
    """The tcgen05 kernel alone (bf16, d=128, C=64), several chunks with and
    without a ragged tail, with a random initial state."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=T, H=3)
    check_fwd(inp, "tc")


def test_two_kernel_forward_is_deterministic():
    """The pre-pass hands chunk-heads out through a counter and picks its
    reserved SMs by which TPCs register first, so the schedule differs from
    call to call; every record is still computed by the same arithmetic, so
    repeated calls give bit-identical o and hT (1B layer: the state pass
    starts on the released SMs while the reserved ones finish)."""
    d = to_dev(gen.prefill_inputs(gen.LAYER_1B))
    outs = []
    for _ in range(3):
        o, hT = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"],
                              d["eta"], d["eps"], d["h0"], C=64, algo="tc")
        outs.append((o, hT))
    torch.cuda.synchronize()
    for o, hT in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(hT, outs[0][1])


def test_two_kernel_forward_with_more_state_ctas_than_sms():
    """B * H * 2 state-pass CTAs above the SM count: no SM is released, the
    pre-pass runs to the end on every SM and the state pass reads the
    records by their flags as its CTAs find room (B 8, H 16: 256 CTAs)."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=8, T=200, H=16)
    check_fwd(inp, "tc")


def test_tensor_core_and_cuda_core_paths_agree():
    inp = gen.prefill_inputs(gen.LONG_CTX, B=1, T=640, H=2)
    o1, h1 = run_fwd(inp, "tc")
    o2, h2 = run_fwd(inp, "simt")
    assert rel_err(o1, o2.double().cpu().numpy()) <= 2e-2
    assert rel_err(h1, h2.double().cpu().numpy()) <= 2e-2


def test_tensor_core_zero_initial_state_and_no_hT():
    inp = gen.prefill_inputs(gen.LAYER_340M, B=1, T=130, H=2)
    d = to_dev(inp)
    o, hT = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["eta"],
                          d["eps"], None, C=64, algo="tc", want_state=False)
    torch.cuda.synchronize()
    assert hT is None
    o_ref, _ = oracle_fwd(inp)
    assert rel_err(o, o_ref) <= 2e-2


# ---------------------------------------------------------------- GDN mode

def _gdn_as_kla_eta(inp, b):
    """The learned-step recurrence with step b equals KLA with
    eta = b (||k||^2 + eps) (pinned on the CPU by test_gdn_reduction)."""
    k = inp["k"].double().numpy()
    return b * (np.sum(k * k, -1) + inp["eps"])


@pytest.mark.parametrize("algo,w,sizes", [
    ("tc", gen.LAYER_1B, dict(B=1, T=200, H=2)),
    ("simt", gen.LAYER_1B, dict(B=1, T=200, H=2)),
    ("simt", gen.TINY, dict(B=2, T=50, H=2)),
])
def test_given_step_mode_against_oracle(algo, w, sizes):
    inp = gen.prefill_inputs(w, **sizes)
    rng = np.random.default_rng(5)
    b = rng.uniform(0.0, 0.5, inp["eta"].shape).astype(np.float32)
    d = to_dev(inp)
    o, hT = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"],
                          torch.from_numpy(b).cuda(), d["eps"], d["h0"],
                          C=inp["C"], algo=algo, rule="given")
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.kla_fwd(inp["q"], inp["k"], inp["v"],
                                  inp["log_alpha"],
                                  _gdn_as_kla_eta(inp, b.astype(np.float64)),
                                  inp["eps"], inp["h0"])
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol and rel_err(hT, h_ref) <= tol


def test_given_step_decode():
    from dataclasses import replace
    w = replace(gen.DECODE, B=4, H=2)
    d = gen.decode_inputs(w, steps=3)
    S = d["S0"].cuda()
    S_ref = d["S0"].double().numpy()
    rng = np.random.default_rng(6)
    for t in range(3):
        b = rng.uniform(0.0, 0.5, (4, 2)).astype(np.float32)
        args = [d[n][t] for n in ("q", "k", "v", "log_alpha")]
        o = kla.decode_step(*[a.cuda() for a in args],
                            torch.from_numpy(b).cuda(), S, eps=d["eps"],
                            rule="given")
        k = d["k"][t].double().numpy()
        eta_kla = b * (np.sum(k * k, -1) + d["eps"])
        o_ref, S_ref = oracle.kla_decode_step(*args, eta_kla, d["eps"], S_ref)
        assert rel_err(o, o_ref) <= 2e-2
    torch.cuda.synchronize()
    assert rel_err(S, S_ref) <= 1e-4


def test_golden_worked_example_through_the_library():
    """tests/golden/kla_worked_example_2x2.txt through the C ABI (fp32,
    CUDA-core kernel), zero-padded to dk = dv = 16: the padded key and value
    dims change nothing, so the first two columns must be the hand-worked
    values and the rest zero."""
    from golden.fixtures import worked_example_2x2
    g = worked_example_2x2()
    pad = lambda x: np.concatenate(
        [x, np.zeros(x.shape[:-1] + (14,))], -1).astype(np.float32)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    o, hT = kla.chunk_fwd(dev(pad(g["q"])), dev(pad(g["k"])),
                          dev(pad(g["v"])),
                          dev(g["log_alpha"].astype(np.float32)),
                          dev(g["eta"].astype(np.float32)), g["eps"], None,
                          C=16, algo="simt")
    torch.cuda.synchronize()
    o, hT = o.cpu().double().numpy(), hT.cpu().double().numpy()
    np.testing.assert_allclose(o[..., :2], g["o"], rtol=0, atol=1e-6)
    assert np.all(o[..., 2:] == 0)
    np.testing.assert_allclose(hT[:, :, :2, :2], g["hT"], rtol=0, atol=1e-6)
    hT[:, :, :2, :2] = 0
    assert np.all(hT == 0)



def test_device_wait_timeout_is_reported_then_cleared():
    """The bounded-wait path of the tensor-core state kernel: one CTA whose
    copy-issuing thread issues nothing waits 1 ms on barriers nothing will
    arrive on, takes its abort path and sets the fault word; the next
    kla_device_status reports KLA_ERR_TIMEOUT, the one after KLA_OK, and a
    forward pass afterwards is correct (the context stays usable)."""
    assert kla.device_status() == 0
    assert kla.selftest_wait_timeout() == 0
    assert kla.device_status() == -4          # KLA_ERR_TIMEOUT
    assert kla.device_status() == 0
    check_fwd(gen.prefill_inputs(gen.LAYER_1B, B=1, T=130, H=2), "tc")


def test_two_kernel_and_fused_tensor_core_paths_agree():
    """The two tensor-core forward paths (pre-pass + state pass, and the
    single fused kernel) on the same inputs: both within the bf16 bound of
    the oracle, and within it of each other."""
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=300, H=3)
    o2, h2 = run_fwd(inp, "tc")
    of, hf = run_fwd(inp, "tc_fused")
    o_ref, h_ref = oracle_fwd(inp)
    for o, h in ((o2, h2), (of, hf)):
        assert rel_err(o, o_ref) <= 2e-2 and rel_err(h, h_ref) <= 2e-2
    assert rel_err(o2, of.double().cpu().numpy()) <= 2e-2


def test_forward_workspace_and_stream_ordered_scratch_agree():
    """kla_chunk_fwd_ws with a caller workspace and kla_chunk_fwd_ex with
    the library's stream-ordered scratch run the same kernels on the same
    inputs: bit-identical o and hT (the kernels have no atomics)."""
    import ctypes
    inp = gen.prefill_inputs(gen.LAYER_1B, B=2, T=200, H=2)
    d = to_dev(inp)
    o_ws, h_ws = kla.chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"],
                               d["eta"], d["eps"], d["h0"], C=64)
    lib = kla.load_library()
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())
    o = torch.empty_like(o_ws)
    hT = torch.empty_like(h_ws)
    B, T, H, dk = inp["k"].shape
    st = lib.kla_chunk_fwd_ex(P(d["q"]), P(d["k"]), P(d["v"]),
                              P(d["log_alpha"]), P(d["eta"]),
                              ctypes.c_float(inp["eps"]), P(d["h0"]), P(o),
                              P(hT), B, T, H, dk, dk, 64, 1, 0, 0,
                              ctypes.c_void_p(
                                  torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(o, o_ws) and torch.equal(hT, h_ws)
