"""ctypes binding of libkla.so (argument marshalling only).

Every entry point mirrors a C function of ``include/kla.h`` under the same
name without the ``kla_`` prefix.  Tensors are torch CUDA tensors (torch
provides device memory and the current stream; all arithmetic runs in the
library's kernels).  There is no CPU fallback: without the built library or
without CUDA tensors these functions raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

KLA_OK = 0
STATUS_NAMES = {0: "KLA_OK", -1: "KLA_ERR_INVALID_ARG",
                -2: "KLA_ERR_UNSUPPORTED_SHAPE", -3: "KLA_ERR_CUDA",
                -4: "KLA_ERR_TIMEOUT", -5: "KLA_ERR_NOT_IMPLEMENTED"}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
ALGOS = {"auto": 0, "simt": 1, "tc": 2, "tc_fused": 3}
RULES = {"kaczmarz": 0, "given": 1}

# name -> (restype, argtypes) of every symbol include/kla.h declares
_VP, _FP, _F, _I = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, \
    ctypes.c_int
SIGNATURES = {
    "kla_chunk_fwd": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                           _I, _I, _I, _I, _I, _I, _I, _VP]),
    "kla_chunk_fwd_ex": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                              _I, _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "kla_chunk_fwd_workspace_size": (
        _I, [_I, _I, _I, _I, _I, _I, _I, _I,
             ctypes.POINTER(ctypes.c_size_t)]),
    "kla_chunk_fwd_ws": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                              _I, _I, _I, _I, _I, _I, _I, _I, _I,
                              _VP, ctypes.c_size_t, _VP]),
    "kla_decode_step": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                             _I, _I, _I, _I, _I, _VP]),
    "kla_decode_step_ex": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                                _I, _I, _I, _I, _I, _I, _VP]),
    "kla_chunk_bwd_workspace_size": (_I, [_I, _I, _I, _I, _I, _I,
                                         ctypes.POINTER(ctypes.c_size_t)]),
    "kla_chunk_bwd": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                           _VP, _VP, _VP, _FP, _FP, _FP,
                           _I, _I, _I, _I, _I, _I, _I, _I,
                           _VP, ctypes.c_size_t, _VP]),
    "kla_chunk_bwd_noalloc": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                                   _FP, _VP, _VP, _VP, _FP, _FP, _FP,
                                   _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "kla_precond_keys": (_I, [_VP, _FP, _VP, _FP, _I, _I, _I, _I, _F, _F,
                              _I, _VP]),
    "kla_precond_keys_workspace_size": (
        _I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "kla_precond_keys_ex": (_I, [_VP, _FP, _VP, _FP, _I, _I, _I, _I, _F, _F,
                                 _I, _VP, ctypes.c_size_t, _VP]),
    "kla_chunk_fwd_kw": (_I, [_VP, _VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                              _FP, _I, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "kla_chunk_fwd_kw_ex": (_I, [_VP, _VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                                 _FP, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                 _VP, ctypes.c_size_t, _VP]),
    "kla_decode_step_kw": (_I, [_VP, _VP, _VP, _VP, _FP, _FP, _F, _FP, _VP,
                                _I, _I, _I, _I, _I, _I, _VP]),
    "kla_chunk_fwd_seq_workspace_size": (
        _I, [_I, _I, _I, _I, _I, _I, _I, _I,
             ctypes.POINTER(ctypes.c_size_t)]),
    "kla_chunk_fwd_seq": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                               _I, _I, _I, _I, _I, _I, _I, _I, _I,
                               _VP, ctypes.c_size_t, _VP]),
    "kla_chunk_fwd_host_workspace_size": (
        _I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "kla_chunk_fwd_host": (_I, [_VP, _VP, _VP, _FP, _FP, _F, _FP, _VP, _FP,
                                _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                _VP, ctypes.c_size_t, _VP]),
    "kla_device_status": (_I, [_VP]),
    "kla_selftest_wait_timeout": (_I, [_VP]),
    "kla_status_string": (ctypes.c_char_p, [_I]),
}

_lib = None


class KlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: "
                         f"{status_string(status)}")


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libkla.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    path = _build.LIB
    if not os.path.exists(path):
        raise KlaError("load_library", -5) from FileNotFoundError(path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().kla_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (no CPU fallback)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def chunk_fwd_workspace_size(B, T, H, dk, dv, C, dtype, algo="auto") -> int:
    """Bytes of device workspace ``chunk_fwd`` needs
    (``kla_chunk_fwd_workspace_size``); 0 for paths that need none."""
    n = ctypes.c_size_t(0)
    st = load_library().kla_chunk_fwd_workspace_size(
        B, T, H, dk, dv, int(C), DTYPES[dtype], ALGOS[algo], ctypes.byref(n))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_workspace_size", st)
    return n.value


def forward_path(B, T, H, dk, dv, C, dtype, algo="auto") -> dict:
    """Which forward kernels ``chunk_fwd`` launches for these sizes (with
    16-byte-aligned tensors, as torch allocates them): the name of the
    path, kernel launches per call and the kernel whose DRAM traffic
    dominates."""
    if chunk_fwd_workspace_size(B, T, H, dk, dv, C, dtype, algo) > 0:
        return {"name": "prepass+state", "launches": 2,
                "traffic_key": "kla_prep_kernel+kla_state_kernel"}
    if dtype == torch.bfloat16 and dk == dv == 128 and C == 64 and \
            algo in ("auto", "tc", "tc_fused"):
        return {"name": "fused", "launches": 1,
                "traffic_key": "kla_chunk_tc"}
    return {"name": "simt", "launches": 1, "traffic_key": "kla_chunk_simt"}


def chunk_fwd(q, k, v, log_alpha, eta, eps: float = 1e-6, h0=None,
              C: int = 64, algo: str = "auto", o=None, hT=None,
              want_state: bool = True, stream=None, rule: str = "kaczmarz",
              workspace=None):
    """KLA forward pass (``kla_chunk_fwd_ws``).

    q, k [B,T,H,dk]; v [B,T,H,dv] (fp32 or bf16, same dtype); log_alpha, eta
    [B,T,H] fp32; h0 [B,H,dk,dv] fp32 or None.  Returns (o, hT); hT is None
    when ``want_state`` is False.  ``o``/``hT`` may be passed preallocated.
    ``rule="given"`` uses eta as the step directly (gated DeltaNet).
    ``workspace``: a device uint8 tensor of at least
    ``chunk_fwd_workspace_size`` bytes, allocated here (by torch) when None.
    """
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    if h0 is not None:
        _check_cuda("h0", h0, torch.float32)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = chunk_fwd_workspace_size(B, T, H, dk, dv, C, q.dtype, algo)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace is not None:
        _check_cuda("workspace", workspace, torch.uint8)
    st = load_library().kla_chunk_fwd_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], ALGOS[algo], RULES[rule], _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_ws", st)
    return o, hT


def chunk_fwd_seq_workspace_size(B, T, H, dk, dv, C, dtype,
                                 segments: int = 0) -> int:
    """Bytes of device workspace ``chunk_fwd_seq`` needs."""
    n = ctypes.c_size_t(0)
    st = load_library().kla_chunk_fwd_seq_workspace_size(
        B, T, H, dk, dv, int(C), DTYPES[dtype], int(segments), ctypes.byref(n))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_seq_workspace_size", st)
    return n.value


def chunk_fwd_seq(q, k, v, log_alpha, eta, eps: float = 1e-6, h0=None,
                  C: int = 64, segments: int = 0, o=None, hT=None,
                  want_state: bool = True, workspace=None, stream=None,
                  rule: str = "kaczmarz"):
    """KLA forward pass split along the sequence (``kla_chunk_fwd_seq``):
    for a few long sequences (bf16, dk = dv = 128, C = 64).  Arguments as
    for ``chunk_fwd``; ``segments`` = 0 picks the split; ``workspace``: a
    device uint8 tensor of ``chunk_fwd_seq_workspace_size`` bytes, allocated
    here when None."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    if h0 is not None:
        _check_cuda("h0", h0, torch.float32)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = chunk_fwd_seq_workspace_size(B, T, H, dk, dv, C, q.dtype, segments)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8,
                                device=q.device)
    _check_cuda("workspace", workspace, torch.uint8)
    st = load_library().kla_chunk_fwd_seq(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], RULES[rule], int(segments), _ptr(workspace),
        workspace.numel(), _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_seq", st)
    return o, hT


def _check_host(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def chunk_fwd_host_workspace_size(B, T, H, dk, dv, C, dtype) -> int:
    """Bytes of device workspace ``chunk_fwd_host`` needs."""
    n = ctypes.c_size_t(0)
    st = load_library().kla_chunk_fwd_host_workspace_size(
        B, T, H, dk, dv, int(C), DTYPES[dtype], ctypes.byref(n))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_host_workspace_size", st)
    return n.value


def chunk_fwd_host(q, k, v, log_alpha, eta, eps: float = 1e-6, h0=None,
                   C: int = 64, algo: str = "auto", o=None, hT=None,
                   want_state: bool = True, workspace=None, stream=None,
                   rule: str = "kaczmarz"):
    """KLA forward pass from host tensors to host tensors
    (``kla_chunk_fwd_host``): the copies to and from the device overlap with
    the kernels.  Inputs as for ``chunk_fwd`` but on the host (page-locked
    for the overlap); ``o``/``hT`` are returned on the host (page-locked when
    allocated here) and are valid once ``stream`` (default: the current one)
    has been synchronised.  ``workspace``: a device uint8 tensor of at least
    ``chunk_fwd_host_workspace_size`` bytes, allocated here when None."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_host(n, t, q.dtype)
    _check_host("log_alpha", log_alpha, torch.float32)
    _check_host("eta", eta, torch.float32)
    if h0 is not None:
        _check_host("h0", h0, torch.float32)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype).pin_memory()
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    need = chunk_fwd_host_workspace_size(B, T, H, dk, dv, C, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8,
                                device="cuda")
    _check_cuda("workspace", workspace, torch.uint8)
    st = load_library().kla_chunk_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], ALGOS[algo], RULES[rule], _ptr(workspace),
        workspace.numel(), _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_host", st)
    return o, hT


def decode_step(q, k, v, log_alpha, eta, S, eps: float = 1e-6, o=None,
                stream=None, rule: str = "kaczmarz"):
    """One KLA decode token (``kla_decode_step``); S [N,H,dk,dv] fp32 is
    updated in place.  Returns o [N,H,dv]."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    _check_cuda("S", S, torch.float32)
    N, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    st = load_library().kla_decode_step_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(S), _ptr(o), N, H, dk, dv, DTYPES[q.dtype], RULES[rule],
        _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_decode_step_ex", st)
    return o


def chunk_bwd_workspace_size(B: int, T: int, H: int, dk: int, dv: int,
                             C: int = 64) -> int:
    """Bytes of workspace ``chunk_bwd`` needs (``kla_chunk_bwd_workspace_size``)."""
    n = ctypes.c_size_t(0)
    st = load_library().kla_chunk_bwd_workspace_size(B, T, H, dk, dv, int(C),
                                                     ctypes.byref(n))
    if st != KLA_OK:
        raise KlaError("kla_chunk_bwd_workspace_size", st)
    return int(n.value)


def chunk_bwd(q, k, v, log_alpha, eta, o_grad, hT_grad=None, eps=1e-6,
              h0=None, C: int = 64, rule: str = "kaczmarz", workspace=None,
              want_h0_grad: bool = True, stream=None):
    """Backward pass (``kla_chunk_bwd``): gradients of a loss with respect to
    every input of ``chunk_fwd``, given dL/do (``o_grad``, like o) and dL/dhT
    (``hT_grad``, fp32 [B,H,dk,dv] or None).  Returns a dict with q_grad,
    k_grad, v_grad (input dtype), log_alpha_grad, eta_grad and h0_grad (fp32;
    None unless ``want_h0_grad``).  ``workspace`` may be passed preallocated
    (uint8 CUDA tensor of at least ``chunk_bwd_workspace_size`` bytes).
    """
    for n, t in (("q", q), ("k", k), ("v", v), ("o_grad", o_grad)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    for n, t in (("h0", h0), ("hT_grad", hT_grad)):
        if t is not None:
            _check_cuda(n, t, torch.float32)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    nbytes = chunk_bwd_workspace_size(B, T, H, dk, dv, C)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8,
                                device=q.device)
    _check_cuda("workspace", workspace)
    out = dict(q_grad=torch.empty_like(q), k_grad=torch.empty_like(k),
               v_grad=torch.empty_like(v),
               log_alpha_grad=torch.empty_like(log_alpha),
               eta_grad=torch.empty_like(eta),
               h0_grad=(torch.empty((B, H, dk, dv), dtype=torch.float32,
                                    device=q.device)
                        if want_h0_grad else None))
    st = load_library().kla_chunk_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(h0), _ptr(o_grad), _ptr(hT_grad), _ptr(out["q_grad"]),
        _ptr(out["k_grad"]), _ptr(out["v_grad"]), _ptr(out["log_alpha_grad"]),
        _ptr(out["eta_grad"]), _ptr(out["h0_grad"]), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], RULES[rule], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_chunk_bwd", st)
    return out


def chunk_bwd_noalloc(q, k, v, log_alpha, eta, o_grad, hT_grad=None,
                      eps=1e-6, h0=None, C: int = 64, rule: str = "kaczmarz",
                      want_h0_grad: bool = True, stream=None):
    """``kla_chunk_bwd_noalloc``: as ``chunk_bwd``, with the library's fixed
    32 MiB device array as scratch instead of a workspace (for callers that
    cannot allocate device memory; larger problems raise).  The gradient
    tensors are still allocated here, by torch; a C caller passes its own.
    """
    for n, t in (("q", q), ("k", k), ("v", v), ("o_grad", o_grad)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    for n, t in (("h0", h0), ("hT_grad", hT_grad)):
        if t is not None:
            _check_cuda(n, t, torch.float32)
    if q.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for n, t in (("k", k), ("v", v), ("o_grad", o_grad),
                 ("log_alpha", log_alpha), ("eta", eta), ("h0", h0),
                 ("hT_grad", hT_grad)):
        if t is not None and t.device != q.device:
            raise ValueError(f"{n} is on {t.device}, q on {q.device}")
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    # the library takes the array of the current device and launches there
    with torch.cuda.device(q.device):
        out = dict(q_grad=torch.empty_like(q), k_grad=torch.empty_like(k),
                   v_grad=torch.empty_like(v),
                   log_alpha_grad=torch.empty_like(log_alpha),
                   eta_grad=torch.empty_like(eta),
                   h0_grad=(torch.empty((B, H, dk, dv), dtype=torch.float32,
                                        device=q.device)
                            if want_h0_grad else None))
        st = _bwd_noalloc_call(q, k, v, log_alpha, eta, o_grad, hT_grad, eps,
                               h0, C, rule, out, B, T, H, dk, dv, stream)
    if st != KLA_OK:
        raise KlaError("kla_chunk_bwd_noalloc", st)
    return out


def _bwd_noalloc_call(q, k, v, log_alpha, eta, o_grad, hT_grad, eps, h0, C,
                      rule, out, B, T, H, dk, dv, stream):
    return load_library().kla_chunk_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(eta), float(eps),
        _ptr(h0), _ptr(o_grad), _ptr(hT_grad), _ptr(out["q_grad"]),
        _ptr(out["k_grad"]), _ptr(out["v_grad"]), _ptr(out["log_alpha_grad"]),
        _ptr(out["eta_grad"]), _ptr(out["h0_grad"]), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], RULES[rule], _stream(stream))


def precond_keys_workspace_size(B, T, H, dk, dtype) -> int:
    """Bytes of device workspace ``precond_keys`` takes
    (``kla_precond_keys_workspace_size``); 0 when its kernel needs none."""
    n = ctypes.c_size_t(0)
    st = load_library().kla_precond_keys_workspace_size(
        B, T, H, dk, DTYPES[dtype], ctypes.byref(n))
    if st != KLA_OK:
        raise KlaError("kla_precond_keys_workspace_size", st)
    return n.value


def precond_keys(k, A0=None, x: float = 1.5, delta: float = 1e-6,
                 k_write=None, AT=None, want_AT: bool = True, stream=None,
                 workspace=None):
    """Write keys of the diagonal-preconditioned variant
    (``kla_precond_keys_ex``).  k [B,T,H,dk]; A0 [B,H,dk] fp32 or None.
    ``workspace``: a device buffer of ``precond_keys_workspace_size`` bytes
    or None (allocated here, by torch, when the kernel takes one).
    Returns (k_write, A_T); A_T is None unless ``want_AT``."""
    _check_cuda("k", k)
    if A0 is not None:
        _check_cuda("A0", A0, torch.float32)
    if k.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {k.dtype}")
    B, T, H, dk = k.shape
    if k_write is None:
        k_write = torch.empty_like(k)
    if AT is None and want_AT:
        AT = torch.empty((B, H, dk), dtype=torch.float32, device=k.device)
    need = precond_keys_workspace_size(B, T, H, dk, k.dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=k.device)
    nbytes = 0 if workspace is None else workspace.numel() * \
        workspace.element_size()
    st = load_library().kla_precond_keys_ex(
        _ptr(k), _ptr(A0), _ptr(k_write), _ptr(AT), B, T, H, dk, float(x),
        float(delta), DTYPES[k.dtype], _ptr(workspace), nbytes,
        _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_precond_keys_ex", st)
    return k_write, AT


def chunk_fwd_kw(q, k, k_write, v, log_alpha, eta, eps: float = 1e-6,
                 h0=None, C: int = 64, o=None, hT=None, want_state=True,
                 stream=None, rule: str = "kaczmarz", algo: str = "auto",
                 workspace=None):
    """Forward pass with separate write keys (``kla_chunk_fwd_kw_ex``); see
    ``chunk_fwd`` for the other arguments (``workspace`` as there: allocated
    here, by torch, when the path needs one and none is given)."""
    for n, t in (("q", q), ("k", k), ("k_write", k_write), ("v", v)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    if h0 is not None:
        _check_cuda("h0", h0, torch.float32)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = chunk_fwd_workspace_size(B, T, H, dk, dv, C, q.dtype, algo)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace is not None:
        _check_cuda("workspace", workspace, torch.uint8)
    st = load_library().kla_chunk_fwd_kw_ex(
        _ptr(q), _ptr(k), _ptr(k_write), _ptr(v), _ptr(log_alpha), _ptr(eta),
        float(eps), _ptr(h0), _ptr(o), _ptr(hT), B, T, H, dk, dv, int(C),
        DTYPES[q.dtype], ALGOS[algo], RULES[rule], _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_chunk_fwd_kw_ex", st)
    return o, hT


def decode_step_kw(q, k, k_write, v, log_alpha, eta, S, eps: float = 1e-6,
                   o=None, stream=None, rule: str = "kaczmarz"):
    """One decode token with a separate write key (``kla_decode_step_kw``);
    S [N,H,dk,dv] fp32 is updated in place.  Returns o [N,H,dv]."""
    for n, t in (("q", q), ("k", k), ("k_write", k_write), ("v", v)):
        _check_cuda(n, t, q.dtype)
    _check_cuda("log_alpha", log_alpha, torch.float32)
    _check_cuda("eta", eta, torch.float32)
    _check_cuda("S", S, torch.float32)
    N, H, dk = k.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    st = load_library().kla_decode_step_kw(
        _ptr(q), _ptr(k), _ptr(k_write), _ptr(v), _ptr(log_alpha), _ptr(eta),
        float(eps), _ptr(S), _ptr(o), N, H, dk, dv, DTYPES[q.dtype],
        RULES[rule], _stream(stream))
    if st != KLA_OK:
        raise KlaError("kla_decode_step_kw", st)
    return o


def device_status(stream=None) -> int:
    """``kla_device_status``: sync the stream, read and clear the fault word."""
    return int(load_library().kla_device_status(_stream(stream)))


def selftest_wait_timeout(stream=None) -> int:
    """``kla_selftest_wait_timeout``: one kernel whose device-side waits give
    up after 1 ms (nothing arrives on them); returns the launch status."""
    return int(load_library().kla_selftest_wait_timeout(_stream(stream)))
