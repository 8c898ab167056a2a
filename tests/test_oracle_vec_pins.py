"""Pins the per-channel (vector) decay oracle (oracle.fwd_vec / bwd_vec) to
facts that do not come from it.

The variant: one log-decay per (token, head, key channel) with the pages'
two parameterisations ("Engineering Long-Context Training for
Trillion-Parameter MoE Models: Three Key Breakthroughs", sec. 3.1 speaks of a
per-position cumulative decay; sec. 3.2 gives b*sigmoid(x), b = -5, and
-softplus(x)), so that row i of the dk x dv state decays by its own factor:
    S_t = diag(exp(lambda_t)) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t.
Each pin is chosen so that a plausible slip (a channel index taken from the
wrong operand, the decay applied to the state's columns instead of its rows,
a dropped factor in the decay gradient) fails at least one.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle


def _lam_library(a, b, mode):
    if mode == oracle.BOUNDED:
        return b * expit(a)
    return -np.logaddexp(0.0, a)


def _case(rng, T, H, dk, dv, docs=None, h0=True, a_mean=0.0, a_std=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H, dk)) * a_std + a_mean
    cu = np.array([0, T] if docs is None else docs, dtype=np.int64)
    hh = rng.standard_normal((len(cu) - 1, H, dk, dv)) * 0.5 if h0 else None
    return q, k, v, a, cu, hh


def _brute_force_vec(q, k, v, a, cu, h0, b, mode):
    """O(T^2) closed form with the global cumulative log-decay per channel,
    Gamma_t[i] = sum_{r<=t} lambda_r[i]:
      o_t = sum_i q_t[i] e^{Gamma_t[i]} h0[i,:]
            + sum_{s<=t} (sum_i q_t[i] k_s[i] e^{Gamma_t[i] - Gamma_s[i]}) v_s
      hT  = diag(e^{Gamma_L}) h0 + sum_s (k_s o e^{Gamma_L - Gamma_s}) v_s^T."""
    T, H, dk = q.shape
    dv = v.shape[2]
    lam = _lam_library(a, b, mode)
    o = np.zeros((T, H, dv))
    N = len(cu) - 1
    hT = np.zeros((N, H, dk, dv))
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        for h in range(H):
            G = np.cumsum(lam[s0:s1, h], axis=0)                  # [L, dk]
            Q, K, V = q[s0:s1, h], k[s0:s1, h], v[s0:s1, h]
            L = s1 - s0
            hh = h0[n, h] if h0 is not None else np.zeros((dk, dv))
            if L == 0:
                hT[n, h] = hh
                continue
            # pair weights sum_i q_t[i] k_s[i] e^{G_t[i] - G_s[i]}, causal
            Wts = np.einsum("ti,si,tsi->ts", Q, K, np.exp(G[:, None, :] - G[None, :, :]))
            o[s0:s1, h] = np.tril(Wts) @ V + (Q * np.exp(G)) @ hh
            hT[n, h] = np.exp(G[-1])[:, None] * hh + (K * np.exp(G[-1][None, :] - G)).T @ V
    return o, hT


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_vec_forward_equals_brute_force(mode):
    rng = np.random.default_rng(11)
    q, k, v, a, cu, h0 = _case(rng, 41, 2, 5, 3, docs=[0, 17, 17, 41])
    o, hT = oracle.fwd_vec(q, k, v, a, -5.0, mode, h0=h0, cu_seqlens=cu)
    ro, rhT = _brute_force_vec(q, k, v, a, cu, h0, -5.0, mode)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, rhT, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_vec_with_equal_channels_reduces_to_the_scalar_oracle(mode):
    """Logits equal over the key channels make diag(g_t) = g_t I: the scalar
    recurrence; the decay gradient of the scalar is the sum of the channels'."""
    rng = np.random.default_rng(12)
    q, k, v, a, cu, h0 = _case(rng, 29, 2, 4, 3, docs=[0, 11, 29])
    a_s = a[:, :, 0]
    a_v = np.repeat(a_s[:, :, None], 4, axis=2)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    o_v, hT_v = oracle.fwd_vec(q, k, v, a_v, -5.0, mode, h0=h0, cu_seqlens=cu)
    o_s, hT_s = oracle.fwd(q, k, v, a_s, -5.0, mode, h0=h0, cu_seqlens=cu)
    np.testing.assert_allclose(o_v, o_s, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT_v, hT_s, rtol=1e-13, atol=1e-14)
    gv = oracle.bwd_vec(q, k, v, a_v, dO, -5.0, mode, h0=h0, dhT=dhT, cu_seqlens=cu)
    gs = oracle.bwd(q, k, v, a_s, dO, -5.0, mode, h0=h0, dhT=dhT, cu_seqlens=cu)
    for x, y in zip((gv[0], gv[1], gv[2], gv[4]), (gs[0], gs[1], gs[2], gs[4])):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gv[3].sum(axis=2), gs[3], rtol=1e-11, atol=1e-12)


def test_vec_channels_decay_state_rows_independently():
    """A state with one nonzero row keeps its shape: only that row's channel
    decays it (rows, not columns, of S carry the key channel)."""
    rng = np.random.default_rng(13)
    T, H, dk, dv = 6, 1, 3, 4
    q = rng.standard_normal((T, H, dk))
    k = np.zeros((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H, dk))
    h0 = np.zeros((1, H, dk, dv))
    h0[0, 0, 1] = rng.standard_normal(dv)
    _, hT = oracle.fwd_vec(q, k, v, a, -5.0, oracle.BOUNDED, h0=h0)
    lam = -5.0 * expit(a[:, 0, 1])
    np.testing.assert_allclose(hT[0, 0, 1], math.exp(lam.sum()) * h0[0, 0, 1], rtol=1e-14)
    assert np.all(hT[0, 0, 0] == 0.0) and np.all(hT[0, 0, 2] == 0.0)


def test_vec_b_zero_is_plain_causal_linear_attention():
    rng = np.random.default_rng(14)
    q, k, v, a, cu, h0 = _case(rng, 23, 2, 4, 3)
    o, hT = oracle.fwd_vec(q, k, v, a, 0.0, oracle.BOUNDED, h0=h0)
    S = h0[0].copy()
    for t in range(23):
        S += np.einsum("hi,hj->hij", k[t], v[t])
        np.testing.assert_allclose(o[t], np.einsum("hi,hij->hj", q[t], S), rtol=1e-12, atol=1e-12)
    da = oracle.bwd_vec(q, k, v, a, rng.standard_normal(v.shape), 0.0, oracle.BOUNDED, h0=h0)[3]
    assert np.all(da == 0.0)


def _loss_vec(q, k, v, a, h0, dO, dhT, b, mode, cu):
    o, hT = oracle.fwd_vec(q, k, v, a, b, mode, h0=h0, cu_seqlens=cu)
    return float(np.sum(o * dO) + np.sum(hT * dhT))


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_vec_gradients_match_central_finite_differences(mode):
    rng = np.random.default_rng(15)
    q, k, v, a, cu, h0 = _case(rng, 19, 1, 3, 2, docs=[0, 8, 19], a_std=1.5)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    dq, dk, dv, da, dh0 = oracle.bwd_vec(q, k, v, a, dO, -5.0, mode, h0=h0, dhT=dhT, cu_seqlens=cu,
                                         window=5)
    args = dict(q=q, k=k, v=v, a=a, h0=h0)
    grads = dict(q=dq, k=dk, v=dv, a=da, h0=dh0)
    eps = 1e-6
    for name, x in args.items():
        g = grads[name]
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss_vec(q, k, v, a, h0, dO, dhT, -5.0, mode, cu)
            x[idx] = old - eps
            lm = _loss_vec(q, k, v, a, h0, dO, dhT, -5.0, mode, cu)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-30)
        assert err < 1e-7, f"d{name}: rel err {err:.2e}"


def test_vec_bounded_tile_cumsum_stays_within_the_bound():
    """Per channel the cumulative log-decay over any 16 consecutive tokens
    stays in [16 b, 0]: the reciprocal e^{-Gamma} of every channel is finite
    (the property the bound buys, now channel by channel)."""
    rng = np.random.default_rng(16)
    a = rng.standard_normal((4096, 128)) * 6.0
    lam = oracle.log_decay(a, -5.0, oracle.BOUNDED)
    for s in range(0, 4096, 16):
        G = np.cumsum(lam[s:s + 16], axis=0)
        assert G.min() >= 16 * -5.0 and G.max() <= 0.0
        assert np.all(np.isfinite(np.exp(-G).astype(np.float32)))
