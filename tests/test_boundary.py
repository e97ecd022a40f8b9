"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol ``include/kla.h`` declares, and rejects bad arguments before touching
the device.  No test here launches a kernel (these run without a GPU)."""
import ctypes
import os
import re

import pytest

from linear_attention_delta_gb300 import build as kbuild
from linear_attention_delta_gb300 import kla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kla.h")

INVALID, UNSUPPORTED, OK = -1, -2, 0


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KLA_API\s+[\w\s\*]+?\b(kla_\w+)\s*\(",
                                 text)))


@pytest.fixture(scope="module")
def lib():
    return kla.load_library()


def test_header_declares_expected_entry_points():
    syms = declared_symbols()
    for name in ("kla_chunk_fwd", "kla_chunk_fwd_ex", "kla_decode_step",
                 "kla_decode_step_ex", "kla_chunk_bwd",
                 "kla_chunk_bwd_workspace_size", "kla_device_status",
                 "kla_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and the binding knows the signature of each of them
    assert set(declared_symbols()) <= set(kla.SIGNATURES)


def test_build_is_fresh():
    assert kbuild.up_to_date()


def test_status_strings(lib):
    for code in kla.STATUS_NAMES:
        s = kla.status_string(code)
        assert isinstance(s, str) and s
    assert kla.status_string(12345) == "unknown status"


P = ctypes.c_void_p(0x1000)      # never dereferenced: calls fail validation


def fwd(lib, *, q=P, k=P, v=P, la=P, eta=P, eps=1e-6, h0=None, o=P, hT=None,
        B=1, T=8, H=1, dk=16, dv=16, C=16, dtype=1, algo=0, rule=0):
    return lib.kla_chunk_fwd_ex(q, k, v, la, eta, eps, h0, o, hT, B, T, H, dk,
                                dv, C, dtype, algo, rule, None)


def dec(lib, *, q=P, k=P, v=P, la=P, eta=P, eps=1e-6, S=P, o=P, N=1, H=1,
        dk=16, dv=16, dtype=1):
    return lib.kla_decode_step(q, k, v, la, eta, eps, S, o, N, H, dk, dv,
                               dtype, None)


def test_fwd_rejects_bad_arguments_on_host(lib):
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, o=None) == INVALID
    assert fwd(lib, eta=None) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, T=-3) == INVALID
    assert fwd(lib, C=0) == INVALID
    assert fwd(lib, dtype=7) == INVALID
    assert fwd(lib, algo=9) == INVALID
    assert fwd(lib, rule=2) == INVALID
    assert fwd(lib, eps=-1.0) == INVALID
    assert fwd(lib, eps=float("nan")) == INVALID
    assert fwd(lib, eps=float("inf")) == INVALID
    assert fwd(lib, o=P, q=P) == INVALID                 # o aliases q
    assert fwd(lib, q=ctypes.c_void_p(0x1001)) == INVALID  # misaligned bf16
    assert fwd(lib, dtype=0, v=ctypes.c_void_p(0x1002)) == INVALID


def test_fwd_rejects_unsupported_shapes(lib):
    q, k, v, o = (ctypes.c_void_p(0x1000 * i) for i in (1, 2, 3, 4))
    la, eta = ctypes.c_void_p(0x5000), ctypes.c_void_p(0x6000)
    kw = dict(q=q, k=k, v=v, o=o, la=la, eta=eta)
    assert fwd(lib, dk=24, **kw) == UNSUPPORTED
    assert fwd(lib, dv=256, **kw) == UNSUPPORTED
    assert fwd(lib, C=48, **kw) == UNSUPPORTED
    assert fwd(lib, C=128, **kw) == UNSUPPORTED
    # the tensor-core kernel only takes bf16, dk = dv = 128, C = 64
    assert fwd(lib, algo=2, dtype=0, dk=128, dv=128, C=64, **kw) == UNSUPPORTED
    assert fwd(lib, algo=2, dk=64, dv=64, C=64, **kw) == UNSUPPORTED
    assert fwd(lib, algo=2, dk=128, dv=128, C=32, **kw) == UNSUPPORTED


def test_fwd_empty_batch_is_a_no_op(lib):
    # nothing to compute: returns before any CUDA call, pointers unused
    assert fwd(lib, B=0, q=None, k=None, v=None, la=None, eta=None,
               o=None) == OK
    assert fwd(lib, H=0, q=None, k=None, v=None, la=None, eta=None,
               o=None) == OK


def test_decode_rejects_bad_arguments_on_host(lib):
    assert dec(lib, S=None) == INVALID
    assert dec(lib, N=-1) == INVALID
    assert dec(lib, dtype=3) == INVALID
    assert dec(lib, S=ctypes.c_void_p(0x1004)) == INVALID   # S not 16B aligned
    assert dec(lib, o=P, S=P) == INVALID                     # o aliases S
    assert dec(lib, dk=8) == UNSUPPORTED
    assert dec(lib, eps=-1e-3) == INVALID
    assert dec(lib, N=0, q=None, S=None, o=None) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 1, 16)
    la = torch.zeros(1, 4, 1)
    with pytest.raises(TypeError):
        kla.chunk_fwd(x, x, x, la, la)
    with pytest.raises(TypeError):
        kla.decode_step(x[0], x[0], x[0], la[0], la[0],
                        torch.zeros(4, 1, 16, 16))
    with pytest.raises(TypeError):
        kla.chunk_fwd_seq(x, x, x, la, la)
    with pytest.raises(TypeError):
        kla.chunk_fwd_kw(x, x, x, x, la, la)
    with pytest.raises(TypeError):
        kla.precond_keys(x)


def test_host_binding_checks_its_inputs_before_any_device_call():
    import torch
    x = torch.zeros(1, 4, 1, 16)
    la = torch.zeros(1, 4, 1)
    with pytest.raises(ValueError):          # not contiguous
        kla.chunk_fwd_host(x.transpose(1, 3), x, x, la, la)
    with pytest.raises(TypeError):           # gates must be fp32
        kla.chunk_fwd_host(x, x, x, la.double(), la)
    with pytest.raises(TypeError):           # q, k, v share one dtype
        kla.chunk_fwd_host(x, x.double(), x, la, la)


def bwd(lib, *, ws_bytes=1 << 20, ws=ctypes.c_void_p(0x9000), B=1, T=8, H=1,
        dk=16, dv=16, C=16, dtype=1, rule=0, eps=1e-6, **ptrs):
    names = ["q", "k", "v", "la", "eta", "h0", "g_o", "g_hT", "g_q", "g_k",
             "g_v", "g_la", "g_eta", "g_h0"]
    defaults = {n: ctypes.c_void_p(0x10000 * (i + 1)) for i, n in
                enumerate(names)}
    defaults["h0"] = defaults["g_hT"] = defaults["g_h0"] = None
    defaults.update(ptrs)
    p = [defaults[n] for n in names]
    return lib.kla_chunk_bwd(p[0], p[1], p[2], p[3], p[4], eps, p[5], p[6],
                             p[7], p[8], p[9], p[10], p[11], p[12], p[13],
                             B, T, H, dk, dv, C, dtype, rule, ws, ws_bytes,
                             None)


def test_bwd_workspace_size(lib):
    n = ctypes.c_size_t(0)
    assert lib.kla_chunk_bwd_workspace_size(2, 100, 3, 16, 32, 16,
                                            ctypes.byref(n)) == OK
    assert n.value == 2 * 4 * 2 * 3 * 7 * 16 * 32    # ceil(100/16) = 7
    assert lib.kla_chunk_bwd_workspace_size(2, 100, 3, 16, 32, 0,
                                            ctypes.byref(n)) == INVALID
    assert lib.kla_chunk_bwd_workspace_size(2, 100, 3, 16, 32, 16,
                                            None) == INVALID


def test_bwd_rejects_bad_arguments_on_host(lib):
    assert bwd(lib, q=None) == INVALID
    assert bwd(lib, g_o=None) == INVALID
    assert bwd(lib, g_q=None) == INVALID
    assert bwd(lib, ws=None) == INVALID
    assert bwd(lib, ws_bytes=16) == INVALID                   # too small
    assert bwd(lib, ws=ctypes.c_void_p(0x9008)) == INVALID    # misaligned
    assert bwd(lib, rule=5) == INVALID
    assert bwd(lib, dtype=3) == INVALID
    assert bwd(lib, eps=-1.0) == INVALID
    assert bwd(lib, g_q=ctypes.c_void_p(0x10000)) == INVALID  # aliases q
    assert bwd(lib, g_k=ctypes.c_void_p(0x90000)) == INVALID  # aliases g_q
    assert bwd(lib, dk=24) == UNSUPPORTED
    assert bwd(lib, C=48) == UNSUPPORTED
    assert bwd(lib, B=0, q=None, k=None) == OK                 # empty: no-op


def test_precond_entry_points_reject_bad_arguments_on_host(lib):
    P, Q = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    pk = lib.kla_precond_keys
    assert pk(P, None, Q, None, 1, 8, 2, 16, 1.0, 1e-6, 1, None) == INVALID
    assert pk(P, None, Q, None, 1, 8, 2, 16, 1.5, -1.0, 1, None) == INVALID
    assert pk(P, None, P, None, 1, 8, 2, 16, 1.5, 1e-6, 1, None) == INVALID
    assert pk(P, None, None, None, 1, 8, 2, 16, 1.5, 1e-6, 1, None) == INVALID
    assert pk(P, None, Q, None, 1, 8, 2, 24, 1.5, 1e-6, 1, None) == UNSUPPORTED
    assert pk(None, None, None, None, 0, 8, 2, 16, 1.5, 1e-6, 1, None) == OK
    fk = lib.kla_chunk_fwd_kw
    ptrs = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(10)]
    q, k, kw, v, la, eta, h0, o, hT = ptrs[:9]
    assert fk(q, k, None, v, la, eta, 1e-6, None, o, None, 1, 8, 1, 16, 16,
              16, 1, 0, None) == INVALID                  # no write keys
    assert fk(q, k, o, v, la, eta, 1e-6, None, o, None, 1, 8, 1, 16, 16,
              16, 1, 0, None) == INVALID                  # o aliases k_write
    dk_ = lib.kla_decode_step_kw
    S = ctypes.c_void_p(0x40000)
    assert dk_(q, k, None, v, la, eta, 1e-6, S, o, 1, 1, 16, 16, 1, 0,
               None) == INVALID


def test_precond_workspace_size_and_checks_on_host(lib):
    """kla_precond_keys_ex's chunked form (dk = 128) takes two fp32 rows of
    dk per (batch, head, 64-token chunk), none for a single chunk (T <= 64)
    or another dk; a small, misaligned or overlapping workspace is refused
    before any device call."""
    bf16 = kla.torch.bfloat16
    assert kla.precond_keys_workspace_size(2, 200, 3, 128, bf16) == \
        2 * 3 * 4 * 1024
    assert kla.precond_keys_workspace_size(2, 65, 3, 128, bf16) == \
        2 * 3 * 2 * 1024
    for T in (0, 1, 64):
        assert kla.precond_keys_workspace_size(2, T, 3, 128, bf16) == 0
    assert kla.precond_keys_workspace_size(2, 200, 3, 64, bf16) == 0
    n = ctypes.c_size_t(0)
    ws_size = lib.kla_precond_keys_workspace_size
    assert ws_size(1, 128, 1, 128, 1, None) == INVALID
    assert ws_size(1, -1, 1, 128, 1, ctypes.byref(n)) == INVALID
    assert ws_size(1, 128, 1, 24, 1, ctypes.byref(n)) == UNSUPPORTED
    V = ctypes.c_void_p
    k, kw = 0x100000, 0x200000        # B1 T128 H1 dk128 bf16: 32 KiB each
    need = 2 * 1024                   # two chunks
    assert kla.precond_keys_workspace_size(1, 128, 1, 128, bf16) == need

    def pk(ws, nbytes):
        return lib.kla_precond_keys_ex(V(k), None, V(kw), None, 1, 128, 1,
                                       128, 1.5, 1e-6, 1, V(ws), nbytes,
                                       None)
    assert pk(0x300000, need - 1) == INVALID                 # small
    assert pk(0x300008, need) == INVALID                     # misaligned
    assert pk(k + 0x4000, need) == INVALID                   # inside k
    assert pk(kw + 0x7ff0, need) == INVALID                  # overlaps kw


HP = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(6)]   # distinct


def host_fwd(lib, *, q=HP[0], k=HP[1], v=HP[2], la=HP[3], eta=HP[4],
             eps=1e-6, h0=None, o=HP[5], hT=None, B=1, T=64, H=1, dk=16,
             dv=16, C=16, dtype=0, algo=0, rule=0,
             ws=ctypes.c_void_p(0x10000), ws_bytes=1 << 40):
    return lib.kla_chunk_fwd_host(q, k, v, la, eta, eps, h0, o, hT, B, T, H,
                                  dk, dv, C, dtype, algo, rule, ws, ws_bytes,
                                  None)


def test_host_fwd_workspace_size(lib):
    n = ctypes.c_size_t(123)
    assert lib.kla_chunk_fwd_host_workspace_size(
        4, 4096, 16, 128, 128, 64, 1, ctypes.byref(n)) == OK
    # two slots of one segment (512 tokens: q, k, v, o bf16, two fp32
    # gates), two fp32 states and the forward's own workspace for one
    # segment (that of the default two-kernel path), each rounded up to
    # 256 bytes
    rows = 4 * 512 * 16
    fwd = kla.chunk_fwd_workspace_size(4, 512, 16, 128, 128, 64,
                                       kla.torch.bfloat16)
    fwd = (fwd + 255) // 256 * 256
    assert n.value == (2 * rows * (4 * 128 * 2 + 8) +
                       2 * 4 * 16 * 128 * 128 * 4 + fwd)
    assert lib.kla_chunk_fwd_host_workspace_size(
        0, 64, 3, 16, 16, 16, 0, ctypes.byref(n)) == OK and n.value == 0
    assert lib.kla_chunk_fwd_host_workspace_size(
        1, 64, 1, 24, 16, 16, 0, ctypes.byref(n)) == UNSUPPORTED
    assert lib.kla_chunk_fwd_host_workspace_size(
        1, 64, 1, 16, 16, 16, 0, None) == INVALID
    assert lib.kla_chunk_fwd_host_workspace_size(
        1, -1, 1, 16, 16, 16, 0, ctypes.byref(n)) == INVALID


def test_host_fwd_rejects_bad_arguments_on_host(lib):
    assert host_fwd(lib, ws=None) == INVALID
    assert host_fwd(lib, ws=ctypes.c_void_p(0x10008)) == INVALID   # alignment
    assert host_fwd(lib, ws_bytes=16) == INVALID
    assert host_fwd(lib, q=None) == INVALID
    assert host_fwd(lib, o=None) == INVALID
    assert host_fwd(lib, q=HP[5]) == INVALID            # o aliases q
    assert host_fwd(lib, algo=7) == INVALID
    assert host_fwd(lib, rule=9) == INVALID
    assert host_fwd(lib, eps=-1.0) == INVALID
    assert host_fwd(lib, eps=float("inf")) == INVALID
    assert host_fwd(lib, dk=24) == UNSUPPORTED
    assert host_fwd(lib, C=48) == UNSUPPORTED
    assert host_fwd(lib, B=0) == OK                     # empty: nothing to do


def test_seq_fwd_workspace_size_and_host_checks(lib):
    n = ctypes.c_size_t(7)
    # B1 T131072 H16, two segments
    assert lib.kla_chunk_fwd_seq_workspace_size(
        1, 131072, 16, 128, 128, 64, 1, 2, ctypes.byref(n)) == OK
    st = 1 * 2 * 16 * 128 * 128
    nrec = 16 * (131072 // 64)           # pre-pass records, all chunks
    rec = nrec * 16640 + nrec * 4 + 528   # records, flags, counters
    rec = (rec + 255) // 256 * 256
    assert n.value == (4 * st * 4 + 131072 * 16 * 128 * 2 + st * 2
                       + 64 * 16 * 128 * 2 + rec)
    # one segment: nothing to split, no workspace
    assert lib.kla_chunk_fwd_seq_workspace_size(
        1, 4096, 16, 128, 128, 64, 1, 1, ctypes.byref(n)) == OK
    assert n.value == 0
    for args in ((1, 4096, 16, 64, 64, 64, 1, 2),      # not d128
                 (1, 4096, 16, 128, 128, 64, 0, 2),    # not bf16
                 (1, 4096, 16, 128, 128, 32, 1, 2),    # not C64
                 (1, 4160, 16, 128, 128, 64, 1, 2),    # T not a multiple of 128
                 (1, 4096, 16, 128, 128, 64, 1, 16)):  # P > 8
        assert lib.kla_chunk_fwd_seq_workspace_size(
            *args, ctypes.byref(n)) == UNSUPPORTED, args
    assert lib.kla_chunk_fwd_seq_workspace_size(
        1, 4096, 16, 128, 128, 64, 1, -1, ctypes.byref(n)) == INVALID
    call = lambda **kw: lib.kla_chunk_fwd_seq(
        kw.get("q", HP[0]), HP[1], HP[2], HP[3], HP[4], kw.get("eps", 1e-6),
        None, kw.get("o", HP[5]), None, 1, 4096, 16, 128, 128, 64, 1,
        kw.get("rule", 0), 2, kw.get("ws", ctypes.c_void_p(0x10000)),
        kw.get("ws_bytes", 1 << 40), None)
    assert call(q=None) == INVALID
    assert call(q=HP[5]) == INVALID          # o aliases q
    assert call(rule=5) == INVALID
    assert call(eps=float("nan")) == INVALID
    assert call(ws=None) == INVALID
    assert call(ws_bytes=1024) == INVALID
    assert call(ws=ctypes.c_void_p(0x10010)) == INVALID


def declared_arities():
    """Entry point -> number of parameters, parsed from include/kla.h."""
    text = open(HEADER).read()
    out = {}
    for m in re.finditer(r"KLA_API\s+[\w\s\*]+?\b(kla_\w+)\s*\(([^)]*)\)",
                         text):
        params = [p for p in m.group(2).split(",") if p.strip()]
        if len(params) == 1 and params[0].strip() == "void":
            params = []
        out[m.group(1)] = len(params)
    return out


def test_binding_signatures_match_the_header():
    arities = declared_arities()
    assert set(arities) == set(declared_symbols())
    for name, n in arities.items():
        assert len(kla.SIGNATURES[name][1]) == n, name


def _bufs(n):
    """n distinct fake device addresses 4 GiB apart (never dereferenced)."""
    return [0x10000 + (i << 32) for i in range(n)]


def test_overlapping_buffers_are_refused_on_host(lib):
    """o (and every other written buffer) may not share a byte with an input,
    checked on byte ranges from the sizes rather than start pointers: an o
    that starts inside q, an hT that starts inside h0 without being h0, a
    decode o that runs into S, a gradient that starts inside o_grad."""
    V = ctypes.c_void_p
    q, k, v, la, eta, o, h0, hT = _bufs(8)
    B, T, H, d = 1, 64, 2, 16
    qbytes = B * T * H * d * 2                       # bf16
    # o starting on the last element of q
    assert fwd(lib, q=V(q), k=V(k), v=V(v), la=V(la), eta=V(eta),
               o=V(q + qbytes - 2), B=B, T=T, H=H, dk=d, dv=d) == INVALID
    # hT starting 4 bytes into h0: refused (hT == h0 exactly is allowed)
    assert fwd(lib, q=V(q), k=V(k), v=V(v), la=V(la), eta=V(eta), o=V(o),
               h0=V(h0), hT=V(h0 + 4), B=B, T=T, H=H, dk=d, dv=d) == INVALID
    # hT inside k
    assert fwd(lib, q=V(q), k=V(k), v=V(v), la=V(la), eta=V(eta), o=V(o),
               hT=V(k + 64), B=B, T=T, H=H, dk=d, dv=d) == INVALID
    # decode: o running into S, S running into v
    N, Hd = 2, 2
    S = h0
    assert dec(lib, q=V(q), k=V(k), v=V(v), la=V(la), eta=V(eta), S=V(S),
               o=V(S - 16), N=N, H=Hd) == INVALID
    assert dec(lib, q=V(q), k=V(k), v=V(v), la=V(la), eta=V(eta),
               S=V(v + 16), o=V(o), N=N, H=Hd) == INVALID
    # backward: k_grad starting inside o_grad
    b = _bufs(12)
    st = lib.kla_chunk_bwd(V(b[0]), V(b[1]), V(b[2]), V(b[3]), V(b[4]), 1e-6,
                           None, V(b[5]), None, V(b[6]), V(b[5] + 32),
                           V(b[8]), V(b[9]), V(b[10]), None, 1, 64, 2, 16, 16,
                           16, 1, 0, V(b[11]), 1 << 20, None)
    assert st == INVALID


def test_write_key_forward_checks_on_host(lib):
    """kla_chunk_fwd_kw_ex refuses, before any device call, a missing
    k_write, a k_write not aligned to its element type and an o that
    overlaps k_write."""
    V = ctypes.c_void_p
    b = _bufs(12)
    args = lambda kw, o: (V(b[0]), V(b[1]), kw, V(b[3]), V(b[4]), V(b[5]),
                          1e-6, None, o, None, 1, 64, 1, 128, 128, 64, 1, 0,
                          0, None, 0, None)
    assert lib.kla_chunk_fwd_kw_ex(*args(None, V(b[6]))) == INVALID
    assert lib.kla_chunk_fwd_kw_ex(*args(V(b[2] + 1), V(b[6]))) == INVALID
    assert lib.kla_chunk_fwd_kw_ex(*args(V(b[2]), V(b[2] + 256))) == INVALID
    assert lib.kla_chunk_fwd_kw(V(b[0]), V(b[1]), None, V(b[3]), V(b[4]),
                                V(b[5]), 1e-6, None, V(b[6]), None, 1, 64, 1,
                                128, 128, 64, 1, 0, None) == INVALID


def test_forward_workspace_size_and_missing_workspace(lib):
    """The two-kernel tensor-core path needs a 16,640-byte record and a
    4-byte ready flag per (batch, head, 64-token chunk), the flags rounded up
    to 16 bytes, and 528 bytes of work counters; the other paths need none;
    kla_chunk_fwd_ws refuses a missing workspace when one is needed, before
    any device call."""
    n = 2 * 3 * 4
    assert kla.chunk_fwd_workspace_size(2, 200, 3, 128, 128, 64,
                                        kla.torch.bfloat16, "tc") == \
        n * 16640 + (n * 4 + 15) // 16 * 16 + 528
    for algo in ("simt", "tc_fused"):
        assert kla.chunk_fwd_workspace_size(2, 200, 3, 128, 128, 64,
                                            kla.torch.bfloat16, algo) == 0
    assert kla.chunk_fwd_workspace_size(2, 200, 3, 16, 16, 16,
                                        kla.torch.float32) == 0
    V = ctypes.c_void_p
    b = _bufs(8)
    st = lib.kla_chunk_fwd_ws(V(b[0]), V(b[1]), V(b[2]), V(b[3]), V(b[4]),
                              1e-6, None, V(b[5]), None, 1, 64, 1, 128, 128,
                              64, 1, 2, 0, None, 0, None)
    assert st == INVALID
    n = ctypes.c_size_t(0)
    assert lib.kla_chunk_fwd_workspace_size(1, 64, 1, 128, 128, 64, 1, 7,
                                            ctypes.byref(n)) == INVALID
