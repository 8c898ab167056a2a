"""The per-channel decay kernels' evaluation order, restated in fp64 numpy and
checked against the per-channel oracle (a pin of the algebra, not of the
kernels).

Per 16-token tile (the unit of the bound, "Engineering Long-Context Training
for Trillion-Parameter MoE Models: Three Key Breakthroughs", sec. 3.2), with
Gamma the tile-local cumsum of the log-decay per channel and gamma its total:
  forward   O = (q o e^{Gamma}) S_in + tril((q o e^{Gamma})(k o e^{-Gamma})^T) V
            S_out = diag(e^{gamma}) S_in + (k o e^{gamma - Gamma})^T V
  backward  dq = e^{Gamma} o (dO S_in^T + dP (k o e^{-Gamma}))
            dk = e^{-Gamma} o (dP^T (q o e^{Gamma})) + e^{gamma - Gamma} o (V D^T)
            dv = P^T dO + (k o e^{gamma - Gamma}) D
            dlambda_t[i] = sum_{u < t} X_u[i] + sum_{r >= t} Y_r[i] + e^{gamma_i} <S_in[i,:], D[i,:]>
              X_u = Kt_u o (dP^T Qt)_u - Qt_u o (dP Kt)_u + k_u o dk_inter_u
              Y_r = q_r o dq_inter_r
            D <- diag(e^{gamma}) D + (q o e^{Gamma})^T dO
(P, dP the causal products inside the tile, Qt = q o e^{Gamma}, Kt = k o
e^{-Gamma}, D the adjoint of the state at the tile end.)  Every term of the
decay gradient is a sum over the token pairs (s, r) with s < t <= r, the pairs
whose weight holds lambda_t, taken channel by channel: pairs across the tile
start (Y), across the tile end (the kd part of X), across both (the state
term), and inside the tile (the dP part of X, where pairs on the same side of
t cancel exactly in the telescoped sum).  The shorter identity
sum_{r >= t}(q_r dq_r - k_r dk_r) + <S_out, D> equals it in exact arithmetic but
subtracts large, nearly equal terms; the test checks both.
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


def _tile_factors(lam_tile):
    G = np.cumsum(lam_tile, axis=0)          # [n, dk]
    return G, G[-1]


def tile_fwd(q, k, v, a, h0, b, mode):
    """One document, one head: q, k [L, dk], v [L, dv], a [L, dk]."""
    lam = _lam(a, b, mode)
    S = h0.copy()
    o = np.zeros((len(q), v.shape[1]))
    for s0, s1 in _tiles(len(q)):
        G, gam = _tile_factors(lam[s0:s1])
        Qt, Kt, Kh = q[s0:s1] * np.exp(G), k[s0:s1] * np.exp(-G), k[s0:s1] * np.exp(gam - G)
        o[s0:s1] = Qt @ S + np.tril(Qt @ Kt.T) @ v[s0:s1]
        S = np.exp(gam)[:, None] * S + Kh.T @ v[s0:s1]
    return o, S


def tile_bwd(q, k, v, a, dO, h0, dhT, b, mode):
    lam = _lam(a, b, mode)
    tiles = _tiles(len(q))
    states, S = [], h0.copy()
    for s0, s1 in tiles:
        states.append(S)
        G, gam = _tile_factors(lam[s0:s1])
        S = np.exp(gam)[:, None] * S + (k[s0:s1] * np.exp(gam - G)).T @ v[s0:s1]
    D = dhT.copy()
    dq, dk, dv, da = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(a)
    for (s0, s1), S_in in zip(reversed(tiles), reversed(states)):
        G, gam = _tile_factors(lam[s0:s1])
        Qt, Kt, Kh = q[s0:s1] * np.exp(G), k[s0:s1] * np.exp(-G), k[s0:s1] * np.exp(gam - G)
        P = np.tril(Qt @ Kt.T)
        dP = np.tril(dO[s0:s1] @ v[s0:s1].T)
        dq[s0:s1] = np.exp(G) * (dO[s0:s1] @ S_in.T + dP @ Kt)
        k_inter = np.exp(gam - G) * (v[s0:s1] @ D.T)
        dk[s0:s1] = np.exp(-G) * (dP.T @ Qt) + k_inter
        dv[s0:s1] = P.T @ dO[s0:s1] + Kh @ D
        q_inter = np.exp(G) * (dO[s0:s1] @ S_in.T)
        X = Kt * (dP.T @ Qt) - Qt * (dP @ Kt) + k[s0:s1] * k_inter
        Y = q[s0:s1] * q_inter
        before = np.cumsum(X, axis=0) - X                         # sum_{u < t} X_u
        from_t = np.cumsum(Y[::-1], axis=0)[::-1]                 # sum_{r >= t} Y_r
        dl = before + from_t + np.exp(gam) * np.sum(S_in * D, axis=1)
        # the shorter identity gives the same in exact arithmetic
        Xs = q[s0:s1] * dq[s0:s1] - k[s0:s1] * dk[s0:s1]
        cst = np.exp(gam) * np.sum(S_in * D, axis=1) + np.sum(k[s0:s1] * k_inter, axis=0)
        np.testing.assert_allclose(np.cumsum(Xs[::-1], axis=0)[::-1] + cst, dl, rtol=1e-8, atol=1e-10)
        da[s0:s1] = dl * _dlam(a[s0:s1], b, mode)
        D = np.exp(gam)[:, None] * D + Qt.T @ dO[s0:s1]
    return dq, dk, dv, da, D


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
@pytest.mark.parametrize("L", [1, 16, 37, 80])
def test_tile_order_equals_the_per_channel_oracle(mode, L):
    rng = np.random.default_rng(100 + L)
    dk, dv = 6, 5
    q = rng.standard_normal((L, 1, dk)) * 0.5
    k = rng.standard_normal((L, 1, dk)) * 0.5
    v = rng.standard_normal((L, 1, dv))
    a = rng.standard_normal((L, 1, dk)) * 2.0 + (2.0 if mode == oracle.SOFTPLUS else 0.0)
    h0 = rng.standard_normal((1, 1, dk, dv)) * 0.3
    dO = rng.standard_normal((L, 1, dv))
    dhT = rng.standard_normal((1, 1, dk, dv)) * 0.3
    ro, rhT = oracle.fwd_vec(q, k, v, a, -5.0, mode, h0=h0)
    o, hT = tile_fwd(q[:, 0], k[:, 0], v[:, 0], a[:, 0], h0[0, 0], -5.0, mode)
    np.testing.assert_allclose(o, ro[:, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(hT, rhT[0, 0], rtol=1e-9, atol=1e-11)
    rg = oracle.bwd_vec(q, k, v, a, dO, -5.0, mode, h0=h0, dhT=dhT)
    g = tile_bwd(q[:, 0], k[:, 0], v[:, 0], a[:, 0], dO[:, 0], h0[0, 0], dhT[0, 0], -5.0, mode)
    for name, x, y in zip(("dq", "dk", "dv", "da"), g[:4], rg[:4]):
        np.testing.assert_allclose(x, y[:, 0], rtol=1e-8, atol=1e-10, err_msg=name)
    np.testing.assert_allclose(g[4], rg[4][0, 0], rtol=1e-9, atol=1e-11)


def test_bounded_fold_factors_stay_finite_per_channel():
    """The one factor above 1, e^{-Gamma} on the diagonal tile, stays below
    e^{80} for every channel under the bound, so bf16/fp32 operands hold it."""
    rng = np.random.default_rng(7)
    a = rng.standard_normal((160, 128)) * 8.0
    lam = _lam(a, -5.0, oracle.BOUNDED)
    for s0, s1 in _tiles(160):
        G, _ = _tile_factors(lam[s0:s1])
        assert np.exp(-G).max() <= np.exp(80.0) * (1 + 1e-12)
        assert np.all(np.isfinite(np.exp(-G).astype(np.float32)))
