"""The gated delta rule's 16-token tile order, restated in fp64 numpy and
checked against the token-by-token oracle (a pin of the algebra the kernels
follow, not of the kernels).

Multiplying out the projection, the rule S_t = g_t (I - beta_t k_t k_t^T)
S_{t-1} + beta_t k_t v_t^T is gated linear attention with pseudo-values
    delta_t = beta_t (v_t - g_t S_{t-1}^T k_t),   S_t = g_t S_{t-1} + k_t delta_t^T.
Inside a 16-token tile (the unit of the bound, "Engineering Long-Context
Training for Trillion-Parameter MoE Models: Three Key Breakthroughs",
sec. 3.1-3.2) with Gamma the tile-local cumsum of the log-decay, gamma its
total and the folded operands Kp = k o e^{Gamma} (<= 1), Km = k o e^{-Gamma}
(<= e^{80} under the bound), Qp = q o e^{Gamma}, Kh = k o e^{gamma - Gamma}:
    L     = diag(beta) strict_tril(Kp Km^T)       (beta_t e^{Gamma_t - Gamma_s} k_t.k_s)
    T     = (I + L)^{-1} diag(beta)                (unit lower-triangular solve)
    Delta = T V - (T Kp) S_0
    O     = Qp S_0 + tril(Qp Km^T) Delta
    S_C   = e^{gamma} S_0 + Kh^T Delta
The same fold that the bound makes legal for linear attention carries both
the triangular system and the scores.  The backward is this block's reverse
mode; its decay gradient is checked both as the telescoped per-token sum and
against the oracle.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle

C = 16


def _lam(a, b, mode):
    return b * expit(a) if mode == oracle.BOUNDED else -np.logaddexp(0.0, a)


def _dlam(a, b, mode):
    s = expit(a)
    return b * s * (1 - s) if mode == oracle.BOUNDED else -s


def _tiles(L):
    return [(c, min(c + C, L)) for c in range(0, L, C)]


def _fold(q, k, lam):
    G = np.cumsum(lam)
    gam = G[-1]
    eG = np.exp(G)[:, None]
    return G, gam, q * eG, k * eG, k / eG, k * np.exp(gam - G)[:, None]


def tile_fwd_one(q, k, v, lam, beta, S0):
    G, gam, Qp, Kp, Km, Kh = _fold(q, k, lam)
    n = len(q)
    L = beta[:, None] * np.tril(Kp @ Km.T, -1)
    T = np.linalg.solve(np.eye(n) + L, np.diag(beta))
    W = T @ Kp
    Delta = T @ v - W @ S0
    P = np.tril(Qp @ Km.T)
    O = Qp @ S0 + P @ Delta
    S1 = np.exp(gam) * S0 + Kh.T @ Delta
    return O, S1, dict(G=G, gam=gam, Qp=Qp, Kp=Kp, Km=Km, Kh=Kh, L=L, T=T, W=W, Delta=Delta, P=P)


def tile_fwd(q, k, v, a, beta, h0, b, mode):
    lam = _lam(a, b, mode)
    S = h0.copy()
    o = np.zeros((len(q), v.shape[1]))
    for s0, s1 in _tiles(len(q)):
        o[s0:s1], S, _ = tile_fwd_one(q[s0:s1], k[s0:s1], v[s0:s1], lam[s0:s1], beta[s0:s1], S)
    return o, S


def tile_bwd_one(q, k, v, lam, beta, S0, dO, D):
    """Reverse mode of tile_fwd_one.  Returns dq, dk, dv, dlam, dbeta, dS0."""
    _, _, f = tile_fwd_one(q, k, v, lam, beta, S0)
    G, gam, Qp, Kp, Km, Kh = f["G"], f["gam"], f["Qp"], f["Kp"], f["Km"], f["Kh"]
    T, W, Delta, P = f["T"], f["W"], f["Delta"], f["P"]
    n = len(q)
    M = np.eye(n) + f["L"]
    dDelta = P.T @ dO + Kh @ D
    dP = np.tril(dO @ Delta.T)
    dQp = dO @ S0.T + dP @ Km
    dKm = dP.T @ Qp
    dKh = Delta @ D.T
    dS0 = Qp.T @ dO + np.exp(gam) * D - W.T @ dDelta
    dW = -dDelta @ S0.T
    dT = dDelta @ v.T + dW @ Kp.T
    dv = T.T @ dDelta
    dKp = T.T @ dW
    MinvT_dT = np.linalg.solve(M.T, dT)
    dM = -MinvT_dT @ T.T
    dbeta = np.diag(MinvT_dT).copy()
    A = np.tril(Kp @ Km.T, -1)
    dL = np.tril(dM, -1)
    dbeta += np.sum(dL * A, axis=1)
    dA = beta[:, None] * dL
    dKp += dA @ Km
    dKm += dA.T @ Kp
    eG = np.exp(G)[:, None]
    dq = eG * dQp
    dk = eG * dKp + dKm / eG + np.exp(gam - G)[:, None] * dKh
    # per-token exponent adjoints, telescoped into the log-decays
    dG = np.sum(Qp * dQp + Kp * dKp - Km * dKm - Kh * dKh, axis=1)
    dgam = np.exp(gam) * np.sum(S0 * D) + np.sum(Kh * dKh)
    dlam = np.cumsum(dG[::-1])[::-1] + dgam
    return dq, dk, dv, dlam, dbeta, dS0


def tile_bwd(q, k, v, a, beta, dO, h0, dhT, b, mode):
    lam = _lam(a, b, mode)
    tiles = _tiles(len(q))
    states, S = [], h0.copy()
    for s0, s1 in tiles:
        states.append(S)
        _, S, _ = tile_fwd_one(q[s0:s1], k[s0:s1], v[s0:s1], lam[s0:s1], beta[s0:s1], S)
    D = dhT.copy()
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    da, dbeta = np.zeros_like(a), np.zeros_like(beta)
    for (s0, s1), S0 in zip(reversed(tiles), reversed(states)):
        g = tile_bwd_one(q[s0:s1], k[s0:s1], v[s0:s1], lam[s0:s1], beta[s0:s1], S0, dO[s0:s1], D)
        dq[s0:s1], dk[s0:s1], dv[s0:s1] = g[0], g[1], g[2]
        da[s0:s1] = g[3] * _dlam(a[s0:s1], b, mode)
        dbeta[s0:s1] = g[4]
        D = g[5]
    return dq, dk, dv, da, dbeta, D


def tile_bwd_one_pairs(q, k, v, lam, beta, S0, dO, D):
    """The same reverse mode in the order the backward kernel takes it: the
    16 x 16 products from the raw inputs with the pair factors E_ts =
    e^{Gamma_t - Gamma_s} applied separately, and the decay gradient as
    sums that never cancel: over the token pairs (s < r <= t) that cross r
    for the pair terms of P and L, suffix sums of the terms through
    e^{Gamma_t}, prefix sums of the terms through e^{gamma - Gamma_t}, and
    the state term e^{gamma} <S_0, D>."""
    G = np.cumsum(lam)
    gam = G[-1]
    n = len(q)
    eG = np.exp(G)
    w = np.exp(gam - G)
    E = np.tril(np.exp(G[:, None] - G[None, :]))
    A = k @ k.T
    L = beta[:, None] * np.tril(A * E, -1)
    P = np.tril((q @ k.T) * E)
    T = np.linalg.solve(np.eye(n) + L, np.diag(beta))
    M = eG[:, None] * k
    W = T @ M
    Delta = T @ v - W @ S0
    QS = q @ S0
    # adjoints
    dDelta = P.T @ dO + w[:, None] * (k @ D)
    dS0 = q.T @ (eG[:, None] * dO) + np.exp(gam) * D - W.T @ dDelta
    dP = np.tril(dO @ Delta.T)
    dW = -dDelta @ S0.T
    dT = dDelta @ v.T + dW @ M.T
    dv = T.T @ dDelta
    dMm = T.T @ dW
    X = np.linalg.solve((np.eye(n) + L).T, dT)
    dL = -np.tril(X @ T.T, -1)
    dbeta = np.diag(X) + np.sum(dL * np.tril(A * E, -1), axis=1)
    dA = beta[:, None] * dL * E
    dPE = dP * E
    dq = eG[:, None] * (dO @ S0.T) + dPE @ k
    dk = dPE.T @ q + (w[:, None] * Delta) @ D.T + eG[:, None] * dMm + (dA + dA.T) @ k
    # decay gradient
    pair = dP * P + dL * L                       # per pair (t, s): d/dGamma_t, minus d/dGamma_s
    cross = np.array([pair[r:, :r].sum() for r in range(n)])
    single_suffix = eG * np.sum(QS * dO, axis=1) + eG * np.sum(dMm * k, axis=1)
    dw = np.sum(k * (Delta @ D.T), axis=1)       # d loss / d w_t
    before = np.cumsum(w * dw) - w * dw          # sum over t < r
    dlam = cross + np.cumsum(single_suffix[::-1])[::-1] + before + np.exp(gam) * np.sum(S0 * D)
    return dq, dk, dv, dlam, dbeta, dS0


def _case(rng, L, dk=6, dv=5, mode=oracle.BOUNDED):
    q = rng.standard_normal((L, 1, dk)) * 0.5
    k = rng.standard_normal((L, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((L, 1, dv))
    a = rng.standard_normal((L, 1)) * 2.0 + (2.0 if mode == oracle.SOFTPLUS else 0.0)
    beta = rng.uniform(0.05, 0.95, (L, 1))
    h0 = rng.standard_normal((1, 1, dk, dv)) * 0.3
    dO = rng.standard_normal((L, 1, dv))
    dhT = rng.standard_normal((1, 1, dk, dv)) * 0.3
    return q, k, v, a, beta, h0, dO, dhT


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
@pytest.mark.parametrize("L", [1, 16, 37, 80])
def test_delta_tile_order_equals_the_oracle(mode, L):
    rng = np.random.default_rng(300 + L)
    q, k, v, a, beta, h0, dO, dhT = _case(rng, L, mode=mode)
    ro, rhT = oracle.fwd_delta(q, k, v, a, beta, -5.0, mode, h0=h0)
    o, hT = tile_fwd(q[:, 0], k[:, 0], v[:, 0], a[:, 0], beta[:, 0], h0[0, 0], -5.0, mode)
    np.testing.assert_allclose(o, ro[:, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(hT, rhT[0, 0], rtol=1e-9, atol=1e-11)
    rg = oracle.bwd_delta(q, k, v, a, beta, dO, -5.0, mode, h0=h0, dhT=dhT)
    g = tile_bwd(q[:, 0], k[:, 0], v[:, 0], a[:, 0], beta[:, 0], dO[:, 0], h0[0, 0], dhT[0, 0], -5.0, mode)
    for name, x, y in zip(("dq", "dk", "dv", "da", "dbeta"), g[:5], rg[:5]):
        np.testing.assert_allclose(x, y[:, 0], rtol=1e-8, atol=1e-10, err_msg=name)
    np.testing.assert_allclose(g[5], rg[5][0, 0], rtol=1e-9, atol=1e-11)


def test_unit_lower_solve_is_the_nilpotent_product():
    """(I + L)^{-1} for strictly lower-triangular 16 x 16 L equals
    (I - L)(I + L^2)(I + L^4)(I + L^8) exactly (L^16 = 0): the product form a
    kernel may use in place of the row-by-row substitution."""
    rng = np.random.default_rng(31)
    L = np.tril(rng.standard_normal((C, C)) * 0.3, -1)
    I = np.eye(C)
    L2 = L @ L
    L4 = L2 @ L2
    L8 = L4 @ L4
    prod = (I - L) @ (I + L2) @ (I + L4) @ (I + L8)
    np.testing.assert_allclose(prod, np.linalg.inv(I + L), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
@pytest.mark.parametrize("L", [1, 9, 16])
def test_delta_pair_form_of_the_tile_backward(mode, L):
    """The kernel's evaluation order of one tile's reverse mode (raw-input
    products, separate pair factors, non-cancelling decay-gradient sums)
    equals the reverse mode of the tile's forward."""
    rng = np.random.default_rng(400 + L)
    q, k, v, a, beta, h0, dO, dhT = _case(rng, L, mode=mode)
    lam = _lam(a[:, 0], -5.0, mode)
    args = (q[:, 0], k[:, 0], v[:, 0], lam, beta[:, 0], h0[0, 0], dO[:, 0], dhT[0, 0])
    for name, x, y in zip(("dq", "dk", "dv", "dlam", "dbeta", "dS0"), tile_bwd_one_pairs(*args), tile_bwd_one(*args)):
        np.testing.assert_allclose(x, y, rtol=1e-9, atol=1e-11, err_msg=name)
