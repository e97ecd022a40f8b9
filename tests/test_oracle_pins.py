"""Pins of the CPU oracle against what the KLA page and mathematics fix.

Every test here runs on the CPU (no GPU marker).  None of them re-derives the
oracle's own update formula and compares: each checks a property that a wrong
oracle (dropped decay, residual against the undecayed state, misplaced eps,
read-out before the write, a transposed state, a wrong sign) would violate.

Page cited throughout: gist.science/es/paper/2605.08587 ("Atencion Lineal
Kaczmarz"); the same content appears on the German and French versions.
"""
import numpy as np
import pytest
import scipy.optimize
import torch

import oracle

RTOL = 1e-12


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _rand(rng, B, T, H, dk, dv, alpha_on=True, eta=None, eps=1e-3,
          h0=True):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk)) * rng.uniform(0.3, 3.0,
                                                         (B, T, H, 1))
    v = rng.standard_normal((B, T, H, dv))
    la = (-rng.uniform(0.0, 1.5, (B, T, H)) if alpha_on
          else np.zeros((B, T, H)))
    et = rng.uniform(0.05, 0.95, (B, T, H)) if eta is None else np.full(
        (B, T, H), float(eta))
    S0 = rng.standard_normal((B, H, dk, dv)) if h0 else None
    return q, k, v, la, et, eps, S0


# --------------------------------------------------------------------------
# the two oracle implementations agree (C vs NumPy), and decode == forward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dk,dv", [(5, 3), (16, 16), (7, 12)])
def test_c_and_numpy_oracles_agree(dk, dv):
    rng = np.random.default_rng(1)
    args = _rand(rng, 2, 9, 3, dk, dv)
    o1, h1 = oracle.kla_fwd(*args)
    o2, h2 = oracle.kla_fwd_np(*args)
    assert _rel(o1, o2) < RTOL and _rel(h1, h2) < RTOL


def test_decode_steps_reproduce_forward():
    rng = np.random.default_rng(2)
    q, k, v, la, et, eps, S0 = _rand(rng, 3, 6, 2, 4, 5)
    o_ref, h_ref = oracle.kla_fwd(q, k, v, la, et, eps, S0)
    S = S0
    for t in range(6):
        o, S = oracle.kla_decode_step(q[:, t], k[:, t], v[:, t], la[:, t],
                                      et[:, t], eps, S)
        assert _rel(o, o_ref[:, t]) < RTOL
    assert _rel(S, h_ref) < RTOL


# --------------------------------------------------------------------------
# A worked example, derived by hand from the page's formulas
# --------------------------------------------------------------------------

def test_hand_worked_example():
    """dk = dv = 2, two tokens, exact rational arithmetic done by hand.

    h0 = I.
    token 1: alpha = 1/2, k = (2,0), v = (1,1), eta = 1/2, eps = 0, q = (1,1)
      S~ = I/2;  ||k||^2 = 4 -> beta = 1/8;  S~^T k = (1,0) -> e = (0,1)
      beta k e^T = [[0,1/4],[0,0]]  ->  S1 = [[1/2,1/4],[0,1/2]]
      o1 = S1^T q = (1/2, 3/4)
    token 2: alpha = 1, k = (0,1), v = (2,0), eta = 1, eps = 1, q = (0,2)
      ||k||^2 = 1 -> beta = 1/(1+1) = 1/2;  S1^T k = (0,1/2) -> e = (2,-1/2)
      beta k e^T = [[0,0],[1,-1/4]]  ->  S2 = [[1/2,1/4],[1,1/4]]
      o2 = S2^T q = (2, 1/2)
    eps differs between the two tokens here, so the two tokens are run as two
    calls (the second resumes from the first one's final state).
    """
    h0 = np.eye(2)[None, None]
    o1, S1 = oracle.kla_fwd(np.array([1.0, 1.0]).reshape(1, 1, 1, 2),
                            np.array([2.0, 0.0]).reshape(1, 1, 1, 2),
                            np.array([1.0, 1.0]).reshape(1, 1, 1, 2),
                            np.log([[[0.5]]]), np.array([[[0.5]]]), 0.0, h0)
    np.testing.assert_allclose(o1.ravel(), [0.5, 0.75], rtol=0, atol=1e-15)
    np.testing.assert_allclose(S1[0, 0], [[0.5, 0.25], [0.0, 0.5]], atol=1e-15)
    o2, S2 = oracle.kla_fwd(np.array([0.0, 2.0]).reshape(1, 1, 1, 2),
                            np.array([0.0, 1.0]).reshape(1, 1, 1, 2),
                            np.array([2.0, 0.0]).reshape(1, 1, 1, 2),
                            np.zeros((1, 1, 1)), np.ones((1, 1, 1)), 1.0, S1)
    np.testing.assert_allclose(o2.ravel(), [2.0, 0.5], atol=1e-15)
    np.testing.assert_allclose(S2[0, 0], [[0.5, 0.25], [1.0, 0.25]],
                               atol=1e-15)
    # the NumPy oracle on the same two calls
    o1n, S1n = oracle.kla_fwd_np(np.array([1.0, 1.0]).reshape(1, 1, 1, 2),
                                 np.array([2.0, 0.0]).reshape(1, 1, 1, 2),
                                 np.array([1.0, 1.0]).reshape(1, 1, 1, 2),
                                 np.log([[[0.5]]]), np.array([[[0.5]]]), 0.0,
                                 h0)
    np.testing.assert_allclose(S1n[0, 0], [[0.5, 0.25], [0.0, 0.5]],
                               atol=1e-15)


def test_golden_worked_example_fixture():
    """tests/golden/kla_worked_example_2x2.txt: three tokens worked by hand
    (decay, a half step and a relaxed step included); both oracles reproduce
    every output and the final state."""
    from golden.fixtures import worked_example_2x2
    g = worked_example_2x2()
    args = [g[n] for n in ("q", "k", "v", "log_alpha", "eta")]
    for fwd in (oracle.kla_fwd, oracle.kla_fwd_np):
        o, hT = fwd(*args, g["eps"], None)
        np.testing.assert_allclose(o, g["o"], rtol=0, atol=1e-6)
        np.testing.assert_allclose(hT, g["hT"], rtol=0, atol=1e-6)


# --------------------------------------------------------------------------
# Unrelaxed case (eta = 1, eps = 0): the three properties the page states
# (section "Propiedades Clave": orthogonal projection, exact line search,
# normalised gradient step) and the constrained problem of section
# "Derivacion Teorica".
# --------------------------------------------------------------------------

def test_projection_satisfies_constraint_every_token():
    """With eta=1, eps=0 every write solves S_t^T k_t = v_t exactly, also when
    the state decays (alpha != 1) and dk != dv.  Query = key reads it back."""
    rng = np.random.default_rng(3)
    q, k, v, la, et, eps, S0 = _rand(rng, 2, 25, 2, 5, 3, eta=1.0, eps=0.0)
    o, _ = oracle.kla_fwd(k, k, v, la, et, 0.0, S0)        # q := k
    assert _rel(o, v) < 1e-11
    o, _ = oracle.kla_fwd_np(k, k, v, la, et, 0.0, S0)
    assert _rel(o, v) < 1e-11


def test_projection_is_minimum_norm_change():
    """S_1 - S~ is the minimum-Frobenius-norm solution of the constraint
    k^T (S~ + D) = v^T, as returned by LAPACK's least-squares routine."""
    rng = np.random.default_rng(4)
    dk, dv = 6, 4
    for _ in range(5):
        k = rng.standard_normal(dk) * rng.uniform(0.2, 5.0)
        v = rng.standard_normal(dv)
        h0 = rng.standard_normal((dk, dv))
        la = -rng.uniform(0.0, 2.0)
        _, S1 = oracle.kla_fwd(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk),
                               v.reshape(1, 1, 1, dv), np.full((1, 1, 1), la),
                               np.ones((1, 1, 1)), 0.0, h0[None, None])
        S_dec = np.exp(la) * h0
        rhs = (v - S_dec.T @ k)[None, :]                 # 1 x dv
        D_min, *_ = np.linalg.lstsq(k[None, :], rhs, rcond=None)
        assert _rel(S1[0, 0] - S_dec, D_min) < 1e-12
        # any other solution of the constraint is farther from S~
        Z = rng.standard_normal((dk, dv))
        Z -= np.outer(k, k @ Z) / (k @ k)                 # k^T Z = 0
        assert (np.linalg.norm(S1[0, 0] + Z - S_dec) >=
                np.linalg.norm(S1[0, 0] - S_dec))


def test_step_is_exact_line_search():
    """Along the update direction k e^T, the oracle's step minimises the
    per-token loss 0.5 ||(S~ + b k e^T)^T k - v||^2 (scipy's scalar search)."""
    rng = np.random.default_rng(5)
    dk, dv = 7, 3
    for _ in range(5):
        k = rng.standard_normal(dk) * rng.uniform(0.2, 5.0)
        v = rng.standard_normal(dv)
        h0 = rng.standard_normal((dk, dv))
        la = -rng.uniform(0.0, 2.0)
        _, S1 = oracle.kla_fwd(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk),
                               v.reshape(1, 1, 1, dv), np.full((1, 1, 1), la),
                               np.ones((1, 1, 1)), 0.0, h0[None, None])
        S_dec = np.exp(la) * h0
        D = S1[0, 0] - S_dec
        e = v - S_dec.T @ k
        direction = np.outer(k, e)
        b_code = np.sum(D * direction) / np.sum(direction * direction)
        assert _rel(D, b_code * direction) < 1e-12      # moves along k e^T

        def loss(b):
            r = (S_dec + b * direction).T @ k - v
            return 0.5 * float(r @ r)

        res = scipy.optimize.minimize_scalar(loss, bracket=(0.0, 1.0),
                                             tol=1e-14)
        assert abs(b_code - res.x) <= 1e-6 * abs(res.x)
        for f in (0.9, 1.1):
            assert loss(b_code) <= loss(f * b_code)


def test_step_is_normalised_sgd():
    """The write equals S~ - (1/||k||^2) grad_S 0.5||S^T k - v||^2 at S~,
    with the gradient taken by torch autograd."""
    rng = np.random.default_rng(6)
    dk, dv = 5, 6
    for _ in range(5):
        k = rng.standard_normal(dk) * rng.uniform(0.2, 5.0)
        v = rng.standard_normal(dv)
        h0 = rng.standard_normal((dk, dv))
        la = -rng.uniform(0.0, 2.0)
        _, S1 = oracle.kla_fwd(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk),
                               v.reshape(1, 1, 1, dv), np.full((1, 1, 1), la),
                               np.ones((1, 1, 1)), 0.0, h0[None, None])
        S = torch.tensor(np.exp(la) * h0, dtype=torch.float64,
                         requires_grad=True)
        kt = torch.tensor(k)
        vt = torch.tensor(v)
        loss = 0.5 * torch.sum((S.T @ kt - vt) ** 2)
        loss.backward()
        sgd = (S - S.grad / (kt @ kt)).detach().numpy()
        assert _rel(S1[0, 0], sgd) < 1e-12


# --------------------------------------------------------------------------
# Relaxed step: where eta and eps enter
# --------------------------------------------------------------------------

def test_relaxed_residual_shrinks_by_closed_factor():
    """After a write the residual is (1 - eta ||k||^2/(||k||^2+eps)) times the
    residual before it (both against the decayed state).  Pins the placement
    of eta and eps in beta_t = eta_t/(||k_t||^2 + eps)."""
    rng = np.random.default_rng(7)
    dk, dv = 6, 5
    for eps in (0.0, 1e-3, 0.7, 3.0):
        k = rng.standard_normal(dk) * rng.uniform(0.2, 3.0)
        v = rng.standard_normal(dv)
        h0 = rng.standard_normal((dk, dv))
        la = -rng.uniform(0.0, 2.0)
        eta = rng.uniform(0.05, 0.95)
        o, _ = oracle.kla_fwd(k.reshape(1, 1, 1, dk), k.reshape(1, 1, 1, dk),
                              v.reshape(1, 1, 1, dv), np.full((1, 1, 1), la),
                              np.full((1, 1, 1), eta), eps, h0[None, None])
        r_before = np.exp(la) * h0.T @ k - v
        r_after = o.ravel() - v
        n = k @ k
        assert _rel(r_after, (1.0 - eta * n / (n + eps)) * r_before) < 1e-12


def test_gdn_reduction():
    """With eta_t = b_t (||k_t||^2 + eps) the step is the plain learned scalar
    b_t of gated DeltaNet (the rule KLA replaces, section "Declaracion del
    Problema"), here written as GDN's own update S <- alpha S + b k (v - (alpha
    S)^T k)^T."""
    rng = np.random.default_rng(8)
    B, T, H, dk, dv = 1, 12, 2, 4, 3
    q, k, v, la, _, eps, S0 = _rand(rng, B, T, H, dk, dv, eps=0.25)
    b = rng.uniform(0.0, 0.3, (B, T, H))
    eta = b * (np.sum(k * k, -1) + eps)
    o, hT = oracle.kla_fwd(q, k, v, la, eta, eps, S0)
    S = S0.copy()
    o_gdn = np.zeros_like(o)
    for t in range(T):
        for h in range(H):
            Sh = np.exp(la[0, t, h]) * S[0, h]
            kk, vv = k[0, t, h], v[0, t, h]
            Sh = Sh + b[0, t, h] * np.outer(kk, vv - Sh.T @ kk)
            S[0, h] = Sh
            o_gdn[0, t, h] = Sh.T @ q[0, t, h]
    assert _rel(o, o_gdn) < 1e-12 and _rel(hT, S) < 1e-12


def test_write_scales_key_direction_only():
    """With v = 0 and alpha = 1, one write maps S = k x^T + u y^T (u orthogonal
    to k) to (1 - eta||k||^2/(||k||^2+eps)) k x^T + u y^T: the transition
    I - beta k k^T has that eigenvalue along k and 1 elsewhere."""
    rng = np.random.default_rng(9)
    dk, dv = 5, 4
    k = rng.standard_normal(dk)
    u = rng.standard_normal(dk)
    u -= k * (u @ k) / (k @ k)
    x, y = rng.standard_normal(dv), rng.standard_normal(dv)
    eta, eps = 0.6, 0.4
    h0 = np.outer(k, x) + np.outer(u, y)
    _, S1 = oracle.kla_fwd(np.zeros((1, 1, 1, dk)), k.reshape(1, 1, 1, dk),
                           np.zeros((1, 1, 1, dv)), np.zeros((1, 1, 1)),
                           np.full((1, 1, 1), eta), eps, h0[None, None])
    lam = 1.0 - eta * (k @ k) / (k @ k + eps)
    assert _rel(S1[0, 0], lam * np.outer(k, x) + np.outer(u, y)) < 1e-12


# --------------------------------------------------------------------------
# Closed forms and library reductions
# --------------------------------------------------------------------------

def test_one_hot_key_overwrites_one_row():
    """k = c e_j with eta=1, eps=0, alpha=1: row j of S becomes v/c, every
    other row is unchanged, and the query c e_j reads v back."""
    rng = np.random.default_rng(10)
    dk, dv, j, c = 6, 4, 2, 2.5
    h0 = rng.standard_normal((dk, dv))
    k = np.zeros(dk)
    k[j] = c
    v = rng.standard_normal(dv)
    o, S1 = oracle.kla_fwd(k.reshape(1, 1, 1, dk), k.reshape(1, 1, 1, dk),
                           v.reshape(1, 1, 1, dv), np.zeros((1, 1, 1)),
                           np.ones((1, 1, 1)), 0.0, h0[None, None])
    expect = h0.copy()
    expect[j] = v / c
    assert _rel(S1[0, 0], expect) < 1e-15
    assert _rel(o.ravel(), v) < 1e-15


def test_orthogonal_keys_closed_form():
    """Mutually orthogonal keys (T <= dk), eta=1, eps=0, alpha=1: the writes do
    not interfere, S_T = S_0 + sum_i k_i (v_i - S_0^T k_i)^T / ||k_i||^2 and
    S_T^T k_i = v_i for every i."""
    rng = np.random.default_rng(11)
    dk, dv, T = 6, 4, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    K = (Qm.T * rng.uniform(0.3, 4.0, (dk, 1)))[:T]
    V = rng.standard_normal((T, dv))
    h0 = rng.standard_normal((dk, dv))
    _, S = oracle.kla_fwd(np.zeros((1, T, 1, dk)), K.reshape(1, T, 1, dk),
                          V.reshape(1, T, 1, dv), np.zeros((1, T, 1)),
                          np.ones((1, T, 1)), 0.0, h0[None, None])
    expect = h0 + sum(np.outer(K[i], V[i] - h0.T @ K[i]) / (K[i] @ K[i])
                      for i in range(T))
    assert _rel(S[0, 0], expect) < 1e-12
    assert _rel(S[0, 0].T @ K.T, V.T) < 1e-12


def test_cyclic_kaczmarz_converges_to_affine_projection():
    """Kaczmarz's method: cycling eta=1, eps=0, alpha=1 writes over n <= dk
    independent (non-orthogonal) keys converges to the point of
    {S : K S = V} nearest S_0, i.e. S_0 + lstsq(K, V - K S_0) (LAPACK)."""
    rng = np.random.default_rng(12)
    dk, dv, n, sweeps = 8, 3, 5, 400
    K = rng.standard_normal((n, dk)) + 0.5 * rng.standard_normal(dk)
    V = rng.standard_normal((n, dv))
    h0 = rng.standard_normal((dk, dv))
    T = n * sweeps
    Ks = np.tile(K, (sweeps, 1)).reshape(1, T, 1, dk)
    Vs = np.tile(V, (sweeps, 1)).reshape(1, T, 1, dv)
    _, S = oracle.kla_fwd(np.zeros((1, T, 1, dk)), Ks, Vs, np.zeros((1, T, 1)),
                          np.ones((1, T, 1)), 0.0, h0[None, None])
    D, *_ = np.linalg.lstsq(K, V - K @ h0, rcond=None)
    assert _rel(S[0, 0], h0 + D) < 1e-9


def test_eta_zero_is_pure_decay():
    """eta = 0: nothing is written, S_t = (prod_{s<=t} alpha_s) h0 and
    o_t = S_t^T q_t; with alpha = 1 as well, O = Q h0 (one matrix product)."""
    rng = np.random.default_rng(13)
    B, T, H, dk, dv = 2, 10, 2, 4, 5
    q, k, v, la, _, eps, S0 = _rand(rng, B, T, H, dk, dv)
    eta = np.zeros((B, T, H))
    o, hT = oracle.kla_fwd(q, k, v, la, eta, eps, S0)
    decay = np.exp(np.cumsum(la, axis=1))                 # [B,T,H]
    expect_o = decay[..., None] * np.einsum("bthi,bhij->bthj", q, S0)
    assert _rel(o, expect_o) < 1e-12
    assert _rel(hT, decay[:, -1][..., None, None] * S0) < 1e-12
    o1, _ = oracle.kla_fwd(q, k, v, np.zeros_like(la), eta, eps, S0)
    assert _rel(o1, np.einsum("bthi,bhij->bthj", q, S0)) < 1e-12


def test_zero_key_with_zero_eps_writes_nothing():
    """k = 0, eps = 0: beta is taken as 0 (the write k e^T is zero anyway)."""
    rng = np.random.default_rng(14)
    dk, dv = 4, 3
    h0 = rng.standard_normal((dk, dv))
    q = rng.standard_normal(dk)
    la = -0.3
    for fn in (oracle.kla_fwd, oracle.kla_fwd_np):
        o, S = fn(q.reshape(1, 1, 1, dk), np.zeros((1, 1, 1, dk)),
                  np.ones((1, 1, 1, dv)), np.full((1, 1, 1), la),
                  np.ones((1, 1, 1)), 0.0, h0[None, None])
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
        assert _rel(S[0, 0], np.exp(la) * h0) < 1e-15
        assert _rel(o.ravel(), np.exp(la) * h0.T @ q) < 1e-15


def test_chunkwise_dense_solve_matches_recurrence():
    """The chunkwise form the GPU path evaluates, solved here with a general
    LU (numpy.linalg.solve, no forward substitution), reproduces the
    sequential recurrence.  Per chunk with start state S0 and in-chunk
    cumulative log-decay g_r, gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i):
        A = I + strict_lower(Diag(beta) (Gamma o K K^T))
        A U~ = Diag(beta) V - Diag(beta) Diag(gamma) K S0
        O = Diag(gamma) Q S0 + lower_incl(Gamma o Q K^T) U~
        S_C = gamma_C S0 + (Diag(Gamma_{C,.}) K)^T U~
    The only KLA-specific part is B = Diag(beta) (section "Implementacion"
    of the page: the block solver changes only through B)."""
    rng = np.random.default_rng(15)
    B_, H, dk, dv, C = 1, 2, 8, 5, 16
    for T in (16, 48, 40):
        q, k, v, la, et, eps, S0 = _rand(rng, B_, T, H, dk, dv, eps=1e-2)
        o_ref, h_ref = oracle.kla_fwd(q, k, v, la, et, eps, S0)
        o = np.zeros_like(o_ref)
        hT = np.zeros_like(h_ref)
        for h in range(H):
            S = S0[0, h].copy()
            for c0 in range(0, T, C):
                sl = slice(c0, min(c0 + C, T))
                Q, K, V = q[0, sl, h], k[0, sl, h], v[0, sl, h]
                n = K.shape[0]
                beta = et[0, sl, h] / (np.sum(K * K, 1) + eps)
                g = np.cumsum(la[0, sl, h])
                gam = np.exp(g)
                Gam = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))
                Gam = np.tril(Gam)
                A = np.eye(n) + np.tril(beta[:, None] * Gam * (K @ K.T), -1)
                rhs = beta[:, None] * V - (beta * gam)[:, None] * (K @ S)
                U = np.linalg.solve(A, rhs)
                o[0, sl, h] = gam[:, None] * (Q @ S) + (Gam * (Q @ K.T)) @ U
                S = gam[-1] * S + (Gam[-1][:, None] * K).T @ U
            hT[0, h] = S
        assert _rel(o, o_ref) < 1e-11 and _rel(hT, h_ref) < 1e-11


def test_segments_resume_from_final_state():
    """Running [0,T) equals [0,T1) then [T1,T) started from the first
    segment's final state (the state is the whole carried context)."""
    rng = np.random.default_rng(16)
    q, k, v, la, et, eps, S0 = _rand(rng, 2, 20, 3, 5, 4)
    o, hT = oracle.kla_fwd(q, k, v, la, et, eps, S0)
    o1, h1 = oracle.kla_fwd(q[:, :7], k[:, :7], v[:, :7], la[:, :7],
                            et[:, :7], eps, S0)
    o2, h2 = oracle.kla_fwd(q[:, 7:], k[:, 7:], v[:, 7:], la[:, 7:],
                            et[:, 7:], eps, h1)
    assert _rel(np.concatenate([o1, o2], 1), o) < 1e-13
    assert _rel(h2, hT) < 1e-13


def test_value_columns_are_independent():
    """Permuting the value columns of v and h0 permutes o and hT the same way
    (each column of S evolves on its own)."""
    rng = np.random.default_rng(17)
    q, k, v, la, et, eps, S0 = _rand(rng, 1, 11, 2, 4, 6)
    perm = rng.permutation(6)
    o, hT = oracle.kla_fwd(q, k, v, la, et, eps, S0)
    op, hp = oracle.kla_fwd(q, k, v[..., perm], la, et, eps, S0[..., perm])
    assert _rel(op, o[..., perm]) < 1e-14 and _rel(hp, hT[..., perm]) < 1e-14


def test_decode_oracle_shapes_and_state_untouched():
    rng = np.random.default_rng(18)
    N, H, dk, dv = 3, 2, 4, 6
    S = rng.standard_normal((N, H, dk, dv))
    S_copy = S.copy()
    o, S_new = oracle.kla_decode_step(rng.standard_normal((N, H, dk)),
                                      rng.standard_normal((N, H, dk)),
                                      rng.standard_normal((N, H, dv)),
                                      -rng.uniform(0, 1, (N, H)),
                                      rng.uniform(0, 1, (N, H)), 1e-6, S)
    assert o.shape == (N, H, dv) and S_new.shape == S.shape
    assert np.array_equal(S, S_copy)


# ---------------------------------------------------------------- backward

def _bwd_case(seed, B=1, T=70, H=2, dk=4, dv=3, with_h0=True, eps=1e-3):
    """Random inputs plus upstream gradients for L = <dout, o> + <dhT, hT>.
    T = 70 crosses the oracle's 64-token checkpoint boundary."""
    rng = np.random.default_rng(seed)
    q, k, v, la, et, eps, S0 = _rand(rng, B, T, H, dk, dv, eps=eps)
    if not with_h0:
        S0 = None
    dout = rng.standard_normal((B, T, H, dv))
    dhT = rng.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, la=la, eta=et, h0=S0), eps, dout, dhT, rng


def _loss(x, eps, dout, dhT, given):
    """L through the (pinned) forward oracle.  The learned-step rule
    beta = b is the Kaczmarz forward with eta = b (||k||^2 + eps), a
    function of (b, k), so its finite differences carry that chain rule."""
    eta = x["eta"]
    if given:
        eta = x["eta"] * (np.sum(x["k"] ** 2, axis=-1) + eps)
    o, hT = oracle.kla_fwd(x["q"], x["k"], x["v"], x["la"], eta, eps,
                           x["h0"])
    return float(np.sum(o * dout) + np.sum(hT * dhT))


_GRAD = dict(q="dq", k="dk", v="dv", la="dlog_alpha", eta="deta",
             h0="dh0")


@pytest.mark.parametrize("given", [False, True], ids=["kaczmarz", "given"])
@pytest.mark.parametrize("with_h0", [True, False])
def test_backward_matches_finite_differences(given, with_h0):
    """Directional central differences of L (through the forward oracle)
    along random directions of every input equal <grad, direction>."""
    x, eps, dout, dhT, rng = _bwd_case(30 + 2 * given + with_h0,
                                       with_h0=with_h0)
    g = oracle.kla_bwd(x["q"], x["k"], x["v"], x["la"], x["eta"], eps,
                       x["h0"], dout, dhT, given=given)
    for name, val in x.items():
        if val is None:
            continue
        for _ in range(2):
            u = rng.standard_normal(val.shape)
            h = 1e-6
            xp, xm = dict(x), dict(x)
            xp[name], xm[name] = val + h * u, val - h * u
            fd = (_loss(xp, eps, dout, dhT, given) -
                  _loss(xm, eps, dout, dhT, given)) / (2 * h)
            an = float(np.sum(g[_GRAD[name]] * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def _torch_forward(q, k, v, la, eta, eps, h0, given):
    """The recurrence in plain PyTorch fp64 (token loop), for autograd."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = (h0.clone() if h0 is not None else
         torch.zeros(B, H, dk, dv, dtype=torch.float64))
    outs = []
    for t in range(T):
        kt, vt, qt = k[:, t], v[:, t], q[:, t]
        St = torch.exp(la[:, t])[..., None, None] * S
        if given:
            beta = eta[:, t]
        else:
            beta = eta[:, t] / ((kt * kt).sum(-1) + eps)
        e = vt - torch.einsum("bhij,bhi->bhj", St, kt)
        S = St + beta[..., None, None] * kt[..., :, None] * e[..., None, :]
        outs.append(torch.einsum("bhij,bhi->bhj", S, qt))
    return torch.stack(outs, 1), S


@pytest.mark.parametrize("given", [False, True], ids=["kaczmarz", "given"])
def test_backward_matches_autograd(given):
    """Reverse mode of an independent PyTorch fp64 forward (autograd)."""
    x, eps, dout, dhT, _ = _bwd_case(40 + given, T=20, H=3, dk=5, dv=4)
    g = oracle.kla_bwd(x["q"], x["k"], x["v"], x["la"], x["eta"], eps,
                       x["h0"], dout, dhT, given=given)
    tx = {n: torch.tensor(a, requires_grad=True) for n, a in x.items()}
    o, hT = _torch_forward(tx["q"], tx["k"], tx["v"], tx["la"], tx["eta"],
                           eps, tx["h0"], given)
    loss = (o * torch.tensor(dout)).sum() + (hT * torch.tensor(dhT)).sum()
    loss.backward()
    for n, t in tx.items():
        assert _rel(g[_GRAD[n]], t.grad.numpy()) < 1e-11, n


def test_backward_closed_form_without_writes():
    """eta = 0 and alpha = 1: S_t = h0 for every t, o_t = h0^T q_t.  Then
    dq_t = h0 dout_t, dh0 = dhT + sum_t q_t dout_t^T, dv = dk = 0,
    dlog_alpha_t = <D_t, h0> and deta_t = k_t^T D_t (v_t - h0^T k_t) /
    (||k_t||^2 + eps), with D_t = dhT + sum_{s >= t} q_s dout_s^T."""
    x, eps, dout, dhT, _ = _bwd_case(50, T=12, H=2, dk=4, dv=3)
    x["eta"] = np.zeros_like(x["eta"])
    x["la"] = np.zeros_like(x["la"])
    g = oracle.kla_bwd(x["q"], x["k"], x["v"], x["la"], x["eta"], eps,
                       x["h0"], dout, dhT)
    q, k, v, h0 = x["q"], x["k"], x["v"], x["h0"]
    B, T, H, _ = q.shape
    D = dhT.copy()
    for t in range(T - 1, -1, -1):
        D = D + np.einsum("bhi,bhj->bhij", q[:, t], dout[:, t])
        assert _rel(g["dq"][:, t],
                    np.einsum("bhij,bhj->bhi", h0, dout[:, t])) < 1e-13
        assert _rel(g["dlog_alpha"][:, t],
                    np.einsum("bhij,bhij->bh", D, h0)) < 1e-12
        e = v[:, t] - np.einsum("bhij,bhi->bhj", h0, k[:, t])
        de = np.einsum("bhi,bhij,bhj->bh", k[:, t], D, e) / (
            np.sum(k[:, t] ** 2, -1) + eps)
        assert _rel(g["deta"][:, t], de) < 1e-12
    assert _rel(g["dh0"], D) < 1e-13
    assert np.max(np.abs(g["dv"])) == 0.0 and np.max(np.abs(g["dk"])) == 0.0


# ---------------------------------------------------------------- preconditioned

def _pcase(seed, B=1, T=30, H=2, dk=6, dv=4):
    rng = np.random.default_rng(seed)
    q, k, v, la, et, eps, S0 = _rand(rng, B, T, H, dk, dv)
    # anisotropic keys, so that the preconditioner is far from the identity
    k = k * rng.uniform(0.2, 3.0, (1, 1, 1, dk))
    return q, k, v, la, et, eps, S0, rng


@pytest.mark.parametrize("given", [False, True])
def test_precond_reduces_to_plain_rule_as_x_tends_to_one(given):
    """x -> 1 squashes P_t onto the identity: write key = read key, and the
    recurrence is the (pinned) plain one."""
    q, k, v, la, et, eps, S0, _ = _pcase(70 + given)
    o, hT, _, kw = oracle.pkla_fwd(q, k, v, la, et, eps, S0, x=1.0 + 1e-12,
                                   given=given)
    assert _rel(kw, k) < 1e-11
    eta = et * (np.sum(k ** 2, -1) + eps) if given else et
    o_ref, h_ref = oracle.kla_fwd(q, k, v, la, eta, eps, S0)
    assert _rel(o, o_ref) < 1e-9 and _rel(hT, h_ref) < 1e-9


def test_precond_kaczmarz_step_is_an_exact_projection():
    """eta = 1, eps = 0: the preconditioned write still satisfies
    S_t^T k_t = v_t after every token (an oblique projection): with q = k the
    read-out returns v."""
    q, k, v, la, _, _, S0, _ = _pcase(72)
    o, _, _, _ = oracle.pkla_fwd(k, k, v, la, np.ones(la.shape), 0.0, S0)
    assert _rel(o, v) < 1e-12


def test_precond_gain_properties():
    """P_t in [1/x, x]; a larger second moment gives a smaller gain; scaling
    every key leaves P unchanged (the squash is centred on the mean log
    second moment); equal second moments give P = 1."""
    q, k, v, la, et, eps, S0, rng = _pcase(73, T=40, dk=8)
    x = 1.5
    _, _, A, kw = oracle.pkla_fwd(q, k, v, la, et, eps, S0, x=x, delta=0.0)
    P = kw / k
    assert P.min() >= 1 / x - 1e-12 and P.max() <= x + 1e-12
    Acum = np.cumsum(k ** 2, axis=1)
    order_A = np.argsort(Acum[0, -1, 0])
    assert np.all(np.diff(P[0, -1, 0][order_A]) <= 1e-12)
    _, _, _, kw2 = oracle.pkla_fwd(q, 3.0 * k, v, la, et, eps, S0, x=x,
                                   delta=0.0)
    assert _rel(kw2, 3.0 * kw) < 1e-12
    kiso = np.ones_like(k) * rng.choice([-1.0, 1.0], k.shape)
    _, _, _, kw3 = oracle.pkla_fwd(q, kiso, v, la, et, eps, S0, x=x,
                                   delta=0.0)
    assert _rel(kw3, kiso) < 1e-12


def test_precond_segments_resume_with_second_moments():
    """[0, T) equals [0, T1) then [T1, T) started from hT and A_T of the
    first segment (A_t is part of the carried context)."""
    q, k, v, la, et, eps, S0, _ = _pcase(74, T=25)
    o, hT, A, _ = oracle.pkla_fwd(q, k, v, la, et, eps, S0)
    o1, h1, A1, _ = oracle.pkla_fwd(q[:, :9], k[:, :9], v[:, :9], la[:, :9],
                                    et[:, :9], eps, S0)
    o2, h2, A2, _ = oracle.pkla_fwd(q[:, 9:], k[:, 9:], v[:, 9:], la[:, 9:],
                                    et[:, 9:], eps, h1, A0=A1)
    assert _rel(np.concatenate([o1, o2], 1), o) < 1e-13
    assert _rel(h2, hT) < 1e-13 and _rel(A2, A) < 1e-14


def test_precond_golden_squash_value():
    """tests/golden/precond_squash_2d.txt: the gain worked by hand for
    A_1 = (1, 4), x = 1.5 (adjacent page "preconditioned DeltaNet", section
    "Aproximacion Diagonal"; the squash is this library's reading, slope 1
    at z = 0, stated in the fixture).  The oracle's write key and second
    moments match the hand values to 1e-12."""
    from golden.fixtures import precond_squash_2d
    g = precond_squash_2d()
    k = g["k"]
    z = np.zeros((1, 1, 1))
    _, _, A, kw = oracle.pkla_fwd(np.zeros_like(k), k, np.zeros((1, 1, 1, 1)),
                                  z, np.ones((1, 1, 1)), 1e-6, None,
                                  A0=g["A0"], x=g["x"], delta=g["delta"])
    np.testing.assert_allclose(kw, g["kw"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(A, g["AT"], rtol=0, atol=1e-15)


def _gain(A_t, x, delta=0.0):
    """P_t of the oracle for the second moments A_t [dk] (one token with
    k = 1 and A_0 = A_t - 1, so that kw = P_t)."""
    dk = A_t.shape[0]
    k = np.ones((1, 1, 1, dk))
    _, _, _, kw = oracle.pkla_fwd(np.zeros_like(k), k, np.zeros((1, 1, 1, 1)),
                                  np.zeros((1, 1, 1)), np.ones((1, 1, 1)),
                                  1e-6, None, A0=(A_t - 1.0).reshape(1, 1, dk),
                                  x=x, delta=delta)
    return kw.reshape(dk)


def test_precond_gain_is_inverse_second_moment_to_first_order():
    """Near equal second moments the squash is the identity in log space
    (slope 1 at z = 0), so the gain is P_t proportional to Diag(A_t)^{-1}
    to first order, as the page's P_t ~ Diag(A_t)^{-1} says: ln(P_i A_i) is
    the same for every i up to O(z^3) terms, and ln P_i / z_i -> 1 with z_i
    the log of the geometric mean of A over A_i."""
    rng = np.random.default_rng(75)
    dk = 8
    for s in (1e-3, 1e-4):
        lnA = rng.standard_normal(dk) * s
        A_t = 2.0 * np.exp(lnA)
        P = _gain(A_t, 1.5)
        z = np.mean(lnA) - lnA
        # ln x tanh(z / ln x) = z - z^3 / (3 ln^2 x) + ...: the departures
        # from the first-order law are third order in z
        zm, l2x = np.max(np.abs(z)), np.log(1.5) ** 2
        lnPA = np.log(P) + np.log(A_t)
        assert np.ptp(lnPA) < zm ** 3 / l2x + 1e-13, (s, np.ptp(lnPA))
        slope = np.log(P) / z
        assert np.max(np.abs(slope - 1.0)) < zm ** 2 / l2x + 1e-8, (s, slope)


def test_precond_pins_reject_other_slopes():
    """The two pins above tell the reading apart from plausible mistakes in
    the squash: gains computed (here, on the CPU) with the slope ln x at
    z = 0, exp(ln x tanh(z)), or with slope 2, exp(ln x tanh(2 z / ln x)),
    miss the hand value and the first-order law P ~ Diag(A)^{-1}."""
    from golden.fixtures import precond_squash_2d
    g = precond_squash_2d()
    lx = np.log(g["x"])
    z0 = np.log(2.0)          # A_1 = (1, 4): z_0 = ln 2
    planted = {"tanh(z)": lambda z: np.exp(lx * np.tanh(z)),
               "tanh(2z/ln x)": lambda z: np.exp(lx * np.tanh(2 * z / lx))}
    for name, gain in planted.items():
        assert abs(gain(z0) - g["kw"][0, 0, 0, 0]) > 1e-3, name
        s = 1e-4
        z = np.array([s, -s])
        P = gain(z)
        A_t = np.exp(-z)              # log-centred second moments
        lnPA = np.log(P) + np.log(A_t)
        assert np.ptp(lnPA) > 1e-5, name
