"""Pins the gated delta rule oracle (oracle.fwd_delta / bwd_delta) to facts
that do not come from it.

The structure: the "Delta Net-style" model that "Engineering Long-Context
Training for Trillion-Parameter MoE Models: Three Key Breakthroughs"
(sec. 3.1) names beside linear attention, with that page's bounded log-decay
(sec. 3.2) in its gate; the rule is the published gated delta rule ("Gated
Delta Networks: Improving Mamba2 with Delta Rule", 2024) for a dk x dv state
read by o = S^T q:
    S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   g_t = e^{lambda_t}.
Each pin is chosen so that a plausible slip (the decay applied to only one
of the two terms, the projection built from q instead of k, beta applied
twice or not at all, a transposed state in the retrieval, a missing term of
the state adjoint) fails at least one.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _lam_library(a, b, mode):
    if mode == oracle.BOUNDED:
        return b * expit(a)
    return -np.logaddexp(0.0, a)


def _case(rng, T, H, dk, dv, docs=None, h0=True, unit_keys=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H))
    beta = rng.uniform(0.05, 0.95, (T, H))
    cu = np.array([0, T] if docs is None else docs, dtype=np.int64)
    hh = rng.standard_normal((len(cu) - 1, H, dk, dv)) * 0.5 if h0 else None
    return q, k, v, a, beta, cu, hh


def _transition_products(q, k, v, a, beta, cu, h0, b, mode):
    """O(T^2) sum over transition products, no recurrence: with
    A_t = g_t (I - beta_t k_t k_t^T) (dk x dk) and B_t = beta_t k_t v_t^T,
        S_t = A_t A_{t-1} ... A_1 h0 + sum_{s<=t} A_t ... A_{s+1} B_s,
    each product formed afresh for every (t, s)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    g = np.exp(_lam_library(a, b, mode))
    o = np.zeros((T, H, dv))
    N = len(cu) - 1
    hT = np.zeros((N, H, dk, dv))
    I = np.eye(dk)
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        for h in range(H):
            A = [g[t, h] * (I - beta[t, h] * np.outer(k[t, h], k[t, h])) for t in range(s0, s1)]
            hh = h0[n, h] if h0 is not None else np.zeros((dk, dv))
            S = None
            for t in range(s1 - s0):
                P = I.copy()
                for x in range(t, -1, -1):
                    P = P @ A[x]
                S = P @ hh
                for s in range(t + 1):
                    P = I.copy()
                    for x in range(t, s, -1):
                        P = P @ A[x]
                    S = S + P @ (beta[s0 + s, h] * np.outer(k[s0 + s, h], v[s0 + s, h]))
                o[s0 + t, h] = S.T @ q[s0 + t, h]
            hT[n, h] = S if S is not None else hh
    return o, hT


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_delta_forward_equals_transition_products(mode):
    rng = np.random.default_rng(21)
    q, k, v, a, beta, cu, h0 = _case(rng, 13, 2, 4, 3, docs=[0, 6, 6, 13])
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, mode, h0=h0, cu_seqlens=cu)
    ro, rhT = _transition_products(q, k, v, a, beta, cu, h0, -5.0, mode)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, rhT, rtol=1e-11, atol=1e-12)


def test_full_write_with_unit_key_retrieves_the_value():
    """beta_t = 1 and |k_t| = 1: the new state maps k_t to v_t exactly, for any
    decay and any earlier state (S_t^T k_t = g (k - k)^T S + v)."""
    rng = np.random.default_rng(22)
    q, k, v, a, beta, cu, h0 = _case(rng, 9, 3, 6, 5)
    beta[:] = 1.0
    q[:] = k                      # reading with the key written last
    o, _ = oracle.fwd_delta(q, k, v, a, beta, -5.0, oracle.BOUNDED, h0=h0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def test_zero_write_strength_only_decays_the_initial_state():
    rng = np.random.default_rng(23)
    q, k, v, a, beta, cu, h0 = _case(rng, 11, 2, 4, 3)
    beta[:] = 0.0
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, oracle.BOUNDED, h0=h0)
    G = np.cumsum(-5.0 * expit(a), axis=0)              # [T, H]
    want = np.exp(G)[:, :, None] * np.einsum("thi,hij->thj", q, h0[0])
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT[0], np.exp(G[-1])[:, None, None] * h0[0], rtol=1e-12)


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_orthogonal_keys_reduce_to_gated_linear_attention(mode):
    """Keys orthogonal to each other and no initial state: every projection
    (I - beta k k^T) leaves the state (built from earlier keys) unchanged, so
    the rule is the scalar-decay recurrence with values beta_t v_t."""
    rng = np.random.default_rng(24)
    T, H, dk, dv = 6, 2, 8, 3
    q, _, v, a, beta, _, _ = _case(rng, T, H, dk, dv, h0=False)
    k = np.zeros((T, H, dk))
    for h in range(H):
        Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        k[:, h] = (Qm[:, :T] * rng.uniform(0.5, 1.5, T)).T
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, mode)
    ro, rhT = oracle.fwd(q, k, v * beta[:, :, None], a, -5.0, mode)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, rhT, rtol=1e-11, atol=1e-12)


def test_one_token_by_hand():
    q = np.array([[[1.0, 2.0]]])
    k = np.array([[[0.6, 0.8]]])
    v = np.array([[[3.0]]])
    a = np.array([[0.0]])                                  # lambda = -2.5
    beta = np.array([[0.5]])
    h0 = np.array([[[[1.0], [-1.0]]]])                     # S_0 = [1, -1]^T
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, oracle.BOUNDED, h0=h0)
    g = np.exp(-2.5)
    r = 0.6 * 1.0 + 0.8 * -1.0                             # S_0^T k = -0.2
    e = 3.0 - g * r
    S1 = g * np.array([1.0, -1.0]) + 0.5 * np.array([0.6, 0.8]) * e
    np.testing.assert_allclose(hT[0, 0, :, 0], S1, rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], 1.0 * S1[0] + 2.0 * S1[1], rtol=1e-14)


def test_documents_are_independent():
    rng = np.random.default_rng(25)
    q, k, v, a, beta, cu, h0 = _case(rng, 30, 2, 4, 3, docs=[0, 7, 19, 19, 30])
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, oracle.BOUNDED, h0=h0, cu_seqlens=cu)
    for n in range(len(cu) - 1):
        s0, s1 = cu[n], cu[n + 1]
        on, hn = oracle.fwd_delta(q[s0:s1], k[s0:s1], v[s0:s1], a[s0:s1], beta[s0:s1], -5.0,
                                  oracle.BOUNDED, h0=h0[n:n + 1])
        np.testing.assert_array_equal(o[s0:s1], on)
        np.testing.assert_array_equal(hT[n], hn[0])


def _loss(q, k, v, a, beta, h0, dO, dhT, cu, mode):
    o, hT = oracle.fwd_delta(q, k, v, a, beta, -5.0, mode, h0=h0, cu_seqlens=cu)
    return float(np.sum(o * dO) + np.sum(hT * dhT))


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_delta_gradients_match_central_differences(mode):
    rng = np.random.default_rng(26)
    q, k, v, a, beta, cu, h0 = _case(rng, 9, 2, 3, 2, docs=[0, 4, 9])
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    grads = oracle.bwd_delta(q, k, v, a, beta, dO, -5.0, mode, h0=h0, dhT=dhT, cu_seqlens=cu, window=3)
    names = ("q", "k", "v", "a", "beta", "h0")
    args = {"q": q, "k": k, "v": v, "a": a, "beta": beta, "h0": h0}
    eps = 1e-6
    for name, g in zip(names, grads):
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, a, beta, h0, dO, dhT, cu, mode)
            x[idx] = old - eps
            lm = _loss(q, k, v, a, beta, h0, dO, dhT, cu, mode)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_delta_backward_window_does_not_change_the_result():
    """The checkpoint window is an evaluation order only."""
    rng = np.random.default_rng(27)
    q, k, v, a, beta, cu, h0 = _case(rng, 40, 2, 4, 3, docs=[0, 23, 40])
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    g1 = oracle.bwd_delta(q, k, v, a, beta, dO, -5.0, oracle.BOUNDED, h0=h0, dhT=dhT, cu_seqlens=cu, window=1)
    g2 = oracle.bwd_delta(q, k, v, a, beta, dO, -5.0, oracle.BOUNDED, h0=h0, dhT=dhT, cu_seqlens=cu, window=1024)
    for x, y in zip(g1, g2):
        np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-14)
