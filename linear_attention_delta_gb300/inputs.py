"""Seeded synthetic inputs for the KLA forward pass and decode step.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle (tests) are
fed from it, so that each side sees identical inputs.

Value distributions (shapes of the 340M / 1B layers and the long contexts the
KLA page evaluates; gist.science/es/paper/2605.08587, sections "Resultados
Experimentales" and "Eficiencia"):

* keys: direction uniform on the sphere, norm log-uniform in [lo, hi];
  the long-context workload additionally rescales 1% of the (t, h) positions
  of every sequence to norm 10 and a disjoint 1% to norm 0.05;
* queries: N(0, 1) for the tiny fp32 case, unit-norm otherwise;
* values: N(0, 1);
* eta = sigmoid(N(0, 1));  log_alpha = -softplus(N(0, 1) + shift);
* initial state: zero, or N(0, 0.02^2) per entry.

q, k, v are drawn in fp32 and rounded once to the workload dtype; the oracle
reads the rounded values (upcast to fp64).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch (prefill) or number of sequences (decode)
    T: int            # tokens per sequence (prefill) / decode steps
    H: int
    dk: int
    dv: int
    C: int            # chunk length (prefill only)
    dtype: str        # "f32" or "bf16" for q, k, v, o
    q_unit: bool
    k_norm: tuple     # (lo, hi) of the log-uniform key norm
    alpha_shift: float
    h0_std: float     # 0 -> zero initial state
    outlier_frac: float = 0.0  # per kind (norm 10 and norm 0.05)
    eps: float = 1e-6
    unrelaxed: bool = False    # eta = 1, eps = 0, log_alpha = 0
    decode: bool = False


TINY = Workload("tiny-fp32-B1-T64-H2-d16-C16", B=1, T=64, H=2, dk=16, dv=16,
                C=16, dtype="f32", q_unit=False, k_norm=(0.25, 4.0),
                alpha_shift=0.0, h0_std=0.0)
TINY_UNRELAXED = replace(TINY, name="tiny-fp32-unrelaxed", eps=0.0,
                         unrelaxed=True)
LAYER_340M = Workload("layer340m-bf16-B8-T2048-H8-d128-C64", B=8, T=2048, H=8,
                      dk=128, dv=128, C=64, dtype="bf16", q_unit=True,
                      k_norm=(0.5, 2.0), alpha_shift=2.0, h0_std=0.0)
LAYER_1B = Workload("layer1b-bf16-B4-T4096-H16-d128-C64", B=4, T=4096, H=16,
                    dk=128, dv=128, C=64, dtype="bf16", q_unit=True,
                    k_norm=(0.5, 2.0), alpha_shift=2.0, h0_std=0.02)
LONG_CTX = Workload("longctx-bf16-B1-T65536-H16-d128-C64", B=1, T=65536,
                    H=16, dk=128, dv=128, C=64, dtype="bf16", q_unit=True,
                    k_norm=(0.5, 2.0), alpha_shift=2.0, h0_std=0.0,
                    outlier_frac=0.01)
DECODE = Workload("decode-bf16-N256-H16-d128-steps1000", B=256, T=1000, H=16,
                  dk=128, dv=128, C=0, dtype="bf16", q_unit=True,
                  k_norm=(0.5, 2.0), alpha_shift=2.0, h0_std=0.02,
                  decode=True)

# The pages' own efficiency points: a 131K-token prefill, and decode at a
# 32K-token context (state carried from the prefill into the decode steps).
LONG_131K = replace(LONG_CTX, name="longctx-bf16-B1-T131072-H16-d128-C64",
                    T=131072)
HANDOFF_32K = replace(LAYER_1B, name="handoff-bf16-B4-T32768-H16-d128-C64",
                      T=32768, h0_std=0.0)

# Seeds: 1000 + position in this list.
WORKLOADS = [TINY, LAYER_340M, LAYER_1B, LONG_CTX, DECODE, LONG_131K,
             HANDOFF_32K]
SEEDS = {w.name: 1000 + i for i, w in enumerate(WORKLOADS)}
SEEDS[TINY_UNRELAXED.name] = SEEDS[TINY.name]

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _softplus(x):
    return np.logaddexp(0.0, x)


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    n[n == 0] = 1.0
    return x / n


def _keys(rng, shape, lo, hi):
    d = _unit_rows(rng, shape)
    norm = np.exp(rng.uniform(np.log(lo), np.log(hi), size=shape[:-1]))
    return d * norm[..., None].astype(np.float32)


def _cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        TORCH_DTYPE[dtype])


def prefill_inputs(w: Workload, seed: int | None = None, **sizes) -> dict:
    """Inputs of one forward pass as CPU torch tensors.

    ``sizes`` may override B, T, H (same distributions at another size).
    Returns dict(q, k, v, log_alpha, eta, h0 (or None), eps, C, workload).
    """
    w = replace(w, **sizes) if sizes else w
    rng = np.random.default_rng(SEEDS.get(w.name, 1000) if seed is None
                                else seed)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    if w.q_unit:
        q = _unit_rows(rng, (B, T, H, dk))
    else:
        q = rng.standard_normal((B, T, H, dk), dtype=np.float32)
    k = _keys(rng, (B, T, H, dk), *w.k_norm)
    if w.outlier_frac > 0.0:
        n_out = int(w.outlier_frac * T)
        for b in range(B):
            for h in range(H):
                pos = rng.choice(T, size=2 * n_out, replace=False)
                big, small = pos[:n_out], pos[n_out:]
                kb = k[b, big, h]
                k[b, big, h] = kb / np.linalg.norm(kb, axis=-1,
                                                   keepdims=True) * 10.0
                ks = k[b, small, h]
                k[b, small, h] = ks / np.linalg.norm(ks, axis=-1,
                                                     keepdims=True) * 0.05
    v = rng.standard_normal((B, T, H, dv), dtype=np.float32)
    eta = _sigmoid(rng.standard_normal((B, T, H))).astype(np.float32)
    log_alpha = (-_softplus(rng.standard_normal((B, T, H)) + w.alpha_shift)
                 ).astype(np.float32)
    eps = w.eps
    if w.unrelaxed:
        eta = np.ones_like(eta)
        log_alpha = np.zeros_like(log_alpha)
        eps = 0.0
    h0 = None
    if w.h0_std > 0.0:
        h0 = torch.from_numpy((rng.standard_normal((B, H, dk, dv)) *
                               w.h0_std).astype(np.float32))
    return dict(q=_cast(q, w.dtype), k=_cast(k, w.dtype), v=_cast(v, w.dtype),
                log_alpha=torch.from_numpy(log_alpha),
                eta=torch.from_numpy(eta), h0=h0, eps=float(eps), C=w.C,
                workload=w)


def decode_inputs(w: Workload, steps: int, seed: int | None = None,
                  **sizes) -> dict:
    """Per-step decode inputs: q, k [steps,N,H,dk]; v [steps,N,H,dv];
    log_alpha, eta [steps,N,H]; S0 [N,H,dk,dv] fp32 (CPU torch tensors)."""
    w = replace(w, **sizes) if sizes else w
    rng = np.random.default_rng(SEEDS.get(w.name, 1000) if seed is None
                                else seed)
    N, H, dk, dv = w.B, w.H, w.dk, w.dv
    q = _unit_rows(rng, (steps, N, H, dk))
    k = _keys(rng, (steps, N, H, dk), *w.k_norm)
    v = rng.standard_normal((steps, N, H, dv), dtype=np.float32)
    eta = _sigmoid(rng.standard_normal((steps, N, H))).astype(np.float32)
    log_alpha = (-_softplus(rng.standard_normal((steps, N, H)) +
                            w.alpha_shift)).astype(np.float32)
    S0 = (rng.standard_normal((N, H, dk, dv), dtype=np.float32) *
          np.float32(w.h0_std)) if w.h0_std > 0 else np.zeros(
              (N, H, dk, dv), np.float32)
    return dict(q=_cast(q, w.dtype), k=_cast(k, w.dtype), v=_cast(v, w.dtype),
                log_alpha=torch.from_numpy(log_alpha),
                eta=torch.from_numpy(eta), S0=torch.from_numpy(S0),
                eps=float(w.eps), workload=w)
