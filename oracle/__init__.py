"""CPU oracle for Kaczmarz Linear Attention (KLA) -- TEST INFRASTRUCTURE.

This package is the checker the CUDA path is compared against.  Only the test
suite, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline`` leg import
it; the product library never does, and nothing here imports the product.

Two independent implementations of the same definition are provided, both in
fp64:

* ``kla_fwd`` / ``kla_decode_step`` -- the C recurrence in ``kla_oracle.c``
  (OpenMP over (batch, head)), used at every size; ``kla_bwd`` -- its
  reverse mode (gradients of every input), derived token by token;
* ``kla_fwd_np`` / ``kla_decode_step_np`` -- a NumPy loop over tokens,
  vectorised over (batch, head), for small cases.

Definition (gist.science/es/paper/2605.08587, sections "Derivacion Teorica"
and "La Regla de Actualizacion KLA"; identical formulas in the German and
French versions of that page):

    S~_{t-1} = alpha_t S_{t-1},             alpha_t = exp(log_alpha_t)
    beta_t   = eta_t / (||k_t||^2 + eps)
    e_t      = v_t - S~_{t-1}^T k_t
    S_t      = S~_{t-1} + beta_t k_t e_t^T
    o_t      = S_t^T q_t

The scalar decay and the read-out are the readings this library adopts (the
pages name a "decayed previous state" but give no formula, and print no
read-out).  beta_t := 0 when ||k_t||^2 + eps == 0.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
the pages and the mathematics fix (projection, exact line search, normalised
SGD step, closed forms, Kaczmarz convergence, a dense solve).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_kla_fwd.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double,
                                       dp, dp, dp,
                                       ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_int]
        lib.oracle_kla_fwd.restype = ctypes.c_int
        lib.oracle_kla_decode_step.argtypes = [dp, dp, dp, dp, dp,
                                               ctypes.c_double, dp, dp,
                                               ctypes.c_long, ctypes.c_long,
                                               ctypes.c_long, ctypes.c_long,
                                               ctypes.c_int]
        lib.oracle_kla_decode_step.restype = ctypes.c_int
        lib.oracle_kla_bwd.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double,
                                       ctypes.c_int, dp, dp, dp,
                                       dp, dp, dp, dp, dp, dp,
                                       ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_int]
        lib.oracle_kla_bwd.restype = ctypes.c_int
        lib.oracle_pkla_fwd.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double,
                                        ctypes.c_int, ctypes.c_double,
                                        ctypes.c_double, dp, dp, dp, dp, dp,
                                        ctypes.c_long, ctypes.c_long,
                                        ctypes.c_long, ctypes.c_long,
                                        ctypes.c_long, ctypes.c_int]
        lib.oracle_pkla_fwd.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Contiguous fp64 copy/view of an array-like (torch tensors included)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    """Threads an OpenMP region of the C oracle uses (1 without OpenMP)."""
    return int(_load().oracle_max_threads())


def kla_fwd(q, k, v, log_alpha, eta, eps, h0=None, n_threads: int = 0):
    """Sequential KLA forward in fp64 (C).

    Shapes: q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha, eta [B,T,H];
    h0 [B,H,dk,dv] or None (zero state).  Returns (o [B,T,H,dv], hT
    [B,H,dk,dv]) as fp64 NumPy arrays.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et = _f64(log_alpha), _f64(eta)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert q.shape == k.shape and v.shape[:3] == (B, T, H)
    assert la.shape == (B, T, H) and et.shape == (B, T, H)
    h0a = None if h0 is None else _f64(h0)
    if h0a is not None:
        assert h0a.shape == (B, H, dk, dv)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = _load().oracle_kla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(et),
                                float(eps), _ptr(h0a), _ptr(o), _ptr(hT),
                                B, T, H, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_kla_fwd failed with {rc}")
    return o, hT


def kla_decode_step(q, k, v, log_alpha, eta, eps, S, n_threads: int = 0):
    """One KLA token for every (sequence, head), fp64 (C).

    Shapes: q, k [N,H,dk]; v [N,H,dv]; log_alpha, eta [N,H]; S [N,H,dk,dv].
    Returns (o [N,H,dv], S_new [N,H,dk,dv]); the input S is not modified.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et = _f64(log_alpha), _f64(eta)
    S = _f64(S).copy()
    N, H, dk = k.shape
    dv = v.shape[-1]
    assert S.shape == (N, H, dk, dv)
    o = np.zeros((N, H, dv), dtype=np.float64)
    rc = _load().oracle_kla_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(la),
                                        _ptr(et), float(eps), _ptr(S), _ptr(o),
                                        N, H, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_kla_decode_step failed with {rc}")
    return o, S


def kla_bwd(q, k, v, log_alpha, eta, eps, h0, dout, dhT=None,
            given: bool = False, n_threads: int = 0) -> dict:
    """Reverse mode of the forward pass in fp64 (C): the gradients of
    L = sum(dout * o) + sum(dhT * hT) with respect to every input.

    ``given=True`` differentiates the learned-step rule beta_t = eta_t
    instead of the Kaczmarz step.  Shapes as in ``kla_fwd``; dout like o,
    dhT like hT (None: zero).  Returns a dict with dq, dk, dv, dlog_alpha,
    deta and dh0 (fp64 NumPy arrays).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et, do = _f64(log_alpha), _f64(eta), _f64(dout)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert q.shape == k.shape and v.shape[:3] == (B, T, H)
    assert la.shape == (B, T, H) and et.shape == (B, T, H)
    assert do.shape == v.shape
    h0a = None if h0 is None else _f64(h0)
    dhTa = None if dhT is None else _f64(dhT)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dlog_alpha=np.zeros_like(la), deta=np.zeros_like(et),
               dh0=np.zeros((B, H, dk, dv)))
    rc = _load().oracle_kla_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(et), float(eps),
        int(bool(given)), _ptr(h0a), _ptr(do), _ptr(dhTa), _ptr(out["dq"]),
        _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dlog_alpha"]),
        _ptr(out["deta"]), _ptr(out["dh0"]), B, T, H, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_kla_bwd failed ({rc})")
    return out


def pkla_fwd(q, k, v, log_alpha, eta, eps, h0=None, A0=None, x=1.5,
             delta=1e-6, given=False, n_threads: int = 0):
    """The diagonal-preconditioned recurrence (write key P_t k_t, P_t from
    the running key second moments squashed into [1/x, x]), fp64 (C).
    Returns (o, hT, A_T, kw) with kw the write keys [B,T,H,dk]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et = _f64(log_alpha), _f64(eta)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    kw = np.zeros((B, T, H, dk))
    A = np.zeros((B, H, dk)) if A0 is None else _f64(A0).copy()
    h0a = None if h0 is None else _f64(h0)
    rc = _load().oracle_pkla_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(et), float(eps),
        int(bool(given)), float(x), float(delta), _ptr(h0a), _ptr(A),
        _ptr(o), _ptr(hT), _ptr(kw), B, T, H, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_pkla_fwd failed ({rc})")
    return o, hT, A, kw


def kla_fwd_np(q, k, v, log_alpha, eta, eps, h0=None):
    """The same recurrence as ``kla_fwd``, as a NumPy fp64 loop over tokens.

    Meant for small inputs; shapes and return values as in ``kla_fwd``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et = _f64(log_alpha), _f64(eta)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv)) if h0 is None else _f64(h0).copy()
    o = np.zeros((B, T, H, dv))
    for t in range(T):
        o[:, t], S = kla_decode_step_np(q[:, t], k[:, t], v[:, t],
                                        la[:, t], et[:, t], eps, S)
    return o, S


def kla_decode_step_np(q, k, v, log_alpha, eta, eps, S):
    """One token for every (n, h) in NumPy fp64; shapes as in
    ``kla_decode_step``.  Returns (o, S_new)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    la, et = _f64(log_alpha), _f64(eta)
    S = _f64(S)
    alpha = np.exp(la)[..., None, None]
    S_dec = alpha * S                                    # decayed state
    denom = np.sum(k * k, axis=-1) + eps
    safe = np.where(denom == 0.0, 1.0, denom)
    beta = np.where(denom == 0.0, 0.0, et / safe)        # Kaczmarz step
    e = v - np.einsum("...ij,...i->...j", S_dec, k)      # residual
    S_new = S_dec + beta[..., None, None] * k[..., :, None] * e[..., None, :]
    o = np.einsum("...ij,...i->...j", S_new, q)          # read-out
    return o, S_new
