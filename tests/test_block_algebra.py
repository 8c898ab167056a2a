"""fp64 restatement of the blocked evaluation order the CUDA kernels use,
checked against the token-by-token oracle.  It pins the algebra (not the
kernels): 128-token blocks made of 16-token decay tiles, every pair weight
built from per-tile factors that are each <= 1 or, on the diagonal tile only,
the tile reciprocal e^{-Gamma} (<= e^{80} with the bound), and the decay
gradient from pair sums.

Per block (block-local cumulative log-decay Lam_t = G_tau + Gamma_t, with
Gamma the tile-local cumsum, gamma_tau the tile total and G_tau the sum of the
tile totals before tile tau inside the block):
  w_ts = e^{Gamma_t} e^{-Gamma_s}                         same tile (s <= t)
  w_ts = e^{Gamma_t} e^{G_tau - G_{sig+1}} e^{gamma_sig - Gamma_s}   sig < tau
  O    = (M o w o Q K^T) V + diag(e^{Lam}) Q S_in
  S_out = e^{Lam_end} S_in + (K o e^{Lam_end - Lam})^T V
Backward per block with E = adjoint of the state at the block end:
  dq = diag(e^{Lam}) dO S_in^T + dP K,      dP = M o w o (dO V^T)
  dk = diag(e^{Lam_end - Lam}) V E^T + dP^T Q
  dv = diag(e^{Lam_end - Lam}) K E + P^T dO, P = M o w o (Q K^T)
  E_prev = e^{Lam_end} E + (Q o e^{Lam})^T dO
  dlam_r = sum_{u<r} X_u + sum_{t>=r} Y_t + e^{Lam_end} <S_in, E>
  X_u = sum_{t>u} W_tu - sum_{s<u} W_us + k_u . dk_inter_u,  Y_t = q_t . dq_inter_t
  W = P o (dO V^T)
"""
import numpy as np
import pytest

import oracle

BT, C = 128, 16


def _lam(a, b, mode):
    return oracle.log_decay(a, b, mode)


def block_weights(lam_blk):
    """Pair weights of one block (length L <= BT) from two-level factors."""
    L = len(lam_blk)
    tile = np.arange(L) // C
    Gam = np.zeros(L)
    for c0 in range(0, L, C):
        Gam[c0:c0 + C] = np.cumsum(lam_blk[c0:c0 + C])
    nt = (L + C - 1) // C
    gam = np.array([Gam[min(c0 + C, L) - 1] for c0 in range(0, L, C)])
    G = np.concatenate([[0.0], np.cumsum(gam)])           # G[tau] = sum of gam before tau
    W = np.zeros((L, L))
    for t in range(L):
        for s in range(t + 1):
            tau, sig = tile[t], tile[s]
            if tau == sig:
                W[t, s] = np.exp(Gam[t]) * np.exp(-Gam[s])
            else:
                W[t, s] = np.exp(Gam[t]) * np.exp(G[tau] - G[sig + 1]) * np.exp(gam[sig] - Gam[s])
    Lam = G[tile] + Gam
    return W, Lam, G[nt]


def blocked_fwd(q, k, v, lam, h0):
    L, dk = q.shape
    S = h0.copy()
    o = np.zeros((L, v.shape[1]))
    for p0 in range(0, L, BT):
        sl = slice(p0, min(p0 + BT, L))
        Wd, Lam, Lend = block_weights(lam[sl])
        Q, K, V = q[sl], k[sl], v[sl]
        o[sl] = (Wd * (Q @ K.T)) @ V + np.exp(Lam)[:, None] * (Q @ S)
        S = np.exp(Lend) * S + (K * np.exp(Lend - Lam)[:, None]).T @ V
    return o, S


def blocked_bwd(q, k, v, lam, h0, dO, dhT):
    L = q.shape[0]
    starts = list(range(0, L, BT))
    Sin = []
    S = h0.copy()
    for p0 in starts:
        Sin.append(S.copy())
        sl = slice(p0, min(p0 + BT, L))
        _, Lam, Lend = block_weights(lam[sl])
        S = np.exp(Lend) * S + (k[sl] * np.exp(Lend - Lam)[:, None]).T @ v[sl]
    E = dhT.copy()
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dlam = np.zeros(L)
    for bi in reversed(range(len(starts))):
        p0 = starts[bi]
        sl = slice(p0, min(p0 + BT, L))
        Wd, Lam, Lend = block_weights(lam[sl])
        Q, K, V, G = q[sl], k[sl], v[sl], dO[sl]
        P = Wd * (Q @ K.T)
        dA = G @ V.T
        dP = Wd * dA
        wk = np.exp(Lend - Lam)
        dq_inter = np.exp(Lam)[:, None] * (G @ Sin[bi].T)
        dk_inter = wk[:, None] * (V @ E.T)
        dv_inter = wk[:, None] * (K @ E)
        dq[sl] = dq_inter + dP @ K
        dk[sl] = dk_inter + dP.T @ Q
        dv[sl] = dv_inter + P.T @ G
        Wp = np.tril(P * dA, -1)
        X = Wp.sum(axis=0) - Wp.sum(axis=1) + np.einsum("ud,ud->u", K, dk_inter)
        Y = np.einsum("td,td->t", Q, dq_inter)
        Cst = np.exp(Lend) * np.sum(Sin[bi] * E)
        n = len(X)
        dlam[sl] = np.concatenate([[0.0], np.cumsum(X)[:-1]]) + np.cumsum(Y[::-1])[::-1] + Cst
        E = np.exp(Lend) * E + (Q * np.exp(Lam)[:, None]).T @ G
        assert n == sl.stop - sl.start
    return dq, dk, dv, dlam, E


@pytest.mark.parametrize("mode,L", [(oracle.BOUNDED, 300), (oracle.BOUNDED, 128), (oracle.SOFTPLUS, 200),
                                    (oracle.BOUNDED, 45)])
def test_blocked_forward_and_backward_equal_recurrence(mode, L):
    rng = np.random.default_rng(L + mode)
    dk, dv, b = 6, 5, -5.0
    q = rng.standard_normal((L, dk)) * 0.4
    k = rng.standard_normal((L, dk)) * 0.4
    v = rng.standard_normal((L, dv))
    a = rng.standard_normal(L) * 2.0 + (2.0 if mode else 0.0)
    h0 = rng.standard_normal((dk, dv)) * 0.3
    dO = rng.standard_normal((L, dv))
    dhT = rng.standard_normal((dk, dv)) * 0.3
    lam = _lam(a, b, mode)
    o, hT = blocked_fwd(q, k, v, lam, h0)
    ro, rhT = oracle.fwd(q[:, None], k[:, None], v[:, None], a[:, None], b, mode, h0=h0[None, None])
    np.testing.assert_allclose(o, ro[:, 0], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(hT, rhT[0, 0], rtol=1e-10, atol=1e-11)
    dq, dk_, dv_, dlam, dh0 = blocked_bwd(q, k, v, lam, h0, dO, dhT)
    rq, rk, rv, rda, rdh0 = oracle.bwd(q[:, None], k[:, None], v[:, None], a[:, None], dO[:, None],
                                       b, mode, h0=h0[None, None], dhT=dhT[None, None])
    np.testing.assert_allclose(dq, rq[:, 0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dk_, rk[:, 0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dv_, rv[:, 0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dh0, rdh0[0, 0], rtol=1e-9, atol=1e-10)
    # dlambda -> da through the decay parameterisation
    s = 1.0 / (1.0 + np.exp(-a))
    dfac = b * s * (1 - s) if mode == oracle.BOUNDED else -s
    np.testing.assert_allclose(dlam * dfac, rda[:, 0], rtol=1e-8, atol=1e-10)


def test_two_level_factors_never_exceed_the_tile_reciprocal():
    """Every factor the blocked order multiplies is <= 1 except the diagonal
    tile's e^{-Gamma_s}, which the bound keeps <= e^{16 |b|} = e^{80}."""
    rng = np.random.default_rng(1)
    lam = _lam(rng.standard_normal(BT) * 4.0 + 3.0, -5.0, oracle.BOUNDED)
    Gam = np.concatenate([np.cumsum(lam[c:c + C]) for c in range(0, BT, C)])
    assert np.all(-Gam <= 80.0 + 1e-12)
    gam = Gam[C - 1::C]
    G = np.concatenate([[0.0], np.cumsum(gam)])
    for tau in range(BT // C):
        for sig in range(tau):
            assert G[tau] - G[sig + 1] <= 0.0
            assert np.all(gam[sig] - Gam[sig * C:(sig + 1) * C] <= 1e-12)


@pytest.mark.parametrize("L", [128, 77])
def test_column_sums_of_w_from_the_pdo_gemm(L):
    """The backward takes the column sums of W = P o dA from the P^T dO GEMM:
    P is causal, so sum_{t>=u} W_tu = v_u . (P^T dO)_u, and
      X_u = v_u . (P^T dO)_u - sum_{s<=u} W_us + k_u . dk_inter_u
    equals the pair-sum form (the diagonal W_uu enters both terms).  The same
    P on both sides (the kernel's bf16 P) keeps every pair inside the block
    cancelling in the prefix sums: sum_{u<r} X_u is then the sum over the
    pairs that cross r, for any P, rounded or not."""
    rng = np.random.default_rng(L)
    dk, dv = 8, 6
    Q, K = rng.standard_normal((L, dk)) * 0.4, rng.standard_normal((L, dk)) * 0.4
    V, G = rng.standard_normal((L, dv)), rng.standard_normal((L, dv))
    E = rng.standard_normal((dk, dv)) * 0.3
    lam = _lam(rng.standard_normal(L), -5.0, oracle.BOUNDED)
    Wd, Lam, Lend = block_weights(lam)
    dA = G @ V.T
    kd = np.einsum("ud,ud->u", K, np.exp(Lend - Lam)[:, None] * (V @ E.T))
    for P in (Wd * (Q @ K.T), np.tril(rng.standard_normal((L, L)))):   # exact, and any causal P
        Wp = np.tril(P * dA, -1)
        X_pairs = Wp.sum(axis=0) - Wp.sum(axis=1) + kd
        X_gemm = np.einsum("ud,ud->u", V, P.T @ G) - np.tril(P * dA).sum(axis=1) + kd
        np.testing.assert_allclose(X_gemm, X_pairs, rtol=1e-10, atol=1e-10)
        W = np.tril(P * dA)
        prefix = np.concatenate([[0.0], np.cumsum(X_gemm - kd)[:-1]])
        crossing = np.array([W[r:, :r].sum() for r in range(L)])
        np.testing.assert_allclose(prefix, crossing, rtol=1e-10, atol=1e-9)
