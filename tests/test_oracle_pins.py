"""Pins the fp64 oracle to facts that do not come from the oracle itself.

Sources of the facts (web pages, cited by title and section):
  "Engineering Long-Context Training for Trillion-Parameter MoE Models: Three
  Key Breakthroughs" sec. 3.1-3.2: chunked linear attention with a per-position
  cumulative decay; log-decay b*sigmoid(x) with b = -5 instead of -softplus(x);
  16-token tiles.
Each pin below is chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, decay applied after instead
of before the update, a wrong derivative of the gate) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, T, H, dk, dv, docs=None, h0=True, a_mean=0.0, a_std=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H)) * a_std + a_mean
    cu = np.array([0, T] if docs is None else docs, dtype=np.int64)
    N = len(cu) - 1
    hh = rng.standard_normal((N, H, dk, dv)) * 0.5 if h0 else None
    return q, k, v, a, cu, hh


def _lam_library(a, b, mode):
    """Log-decay through library routines (scipy expit, numpy logaddexp)."""
    if mode == oracle.BOUNDED:
        return b * expit(a)
    return -np.logaddexp(0.0, a)


def _brute_force(q, k, v, a, cu, h0, b, mode):
    """O(T^2) closed form with the global cumulative log-decay Gamma:
    o_t = e^{Gamma_t} h0^T q_t + sum_{s<=t} e^{Gamma_t - Gamma_s} (q_t.k_s) v_s
    hT  = e^{Gamma_L} h0 + sum_s e^{Gamma_L - Gamma_s} k_s v_s^T."""
    T, H, dk = q.shape
    dv = v.shape[2]
    lam = _lam_library(a, b, mode)
    o = np.zeros((T, H, dv))
    N = len(cu) - 1
    hT = np.zeros((N, H, dk, dv))
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        for h in range(H):
            G = np.cumsum(lam[s0:s1, h])
            Q, K, V = q[s0:s1, h], k[s0:s1, h], v[s0:s1, h]
            L = s1 - s0
            W = np.tril(np.exp(G[:, None] - G[None, :])) * (Q @ K.T)
            o[s0:s1, h] = W @ V
            hh = h0[n, h] if h0 is not None else np.zeros((dk, dv))
            if L:
                o[s0:s1, h] += np.exp(G)[:, None] * (Q @ hh)
                hT[n, h] = math.exp(G[-1]) * hh + (K * np.exp(G[-1] - G)[:, None]).T @ V
            else:
                hT[n, h] = hh
    return o, hT


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_log_decay_matches_library_routines(mode):
    a = np.linspace(-30, 30, 1201)
    lam = oracle.log_decay(a, -5.0, mode)
    np.testing.assert_allclose(lam, _lam_library(a, -5.0, mode), rtol=1e-14, atol=1e-300)


def test_log_decay_special_values():
    # sigmoid(0) = 1/2 and softplus(0) = ln 2 exactly
    assert oracle.log_decay(np.array([0.0]), -5.0, oracle.BOUNDED)[0] == -2.5
    assert abs(oracle.log_decay(np.array([0.0]), -5.0, oracle.SOFTPLUS)[0] + math.log(2)) < 1e-16
    # symmetry: b*sig(x) + b*sig(-x) = b ; softplus(x) - softplus(-x) = x
    x = np.linspace(-20, 20, 81)
    lb = oracle.log_decay(x, -5.0, oracle.BOUNDED) + oracle.log_decay(-x, -5.0, oracle.BOUNDED)
    np.testing.assert_allclose(lb, -5.0, rtol=0, atol=1e-14)
    ls = oracle.log_decay(-x, -5.0, oracle.SOFTPLUS) - oracle.log_decay(x, -5.0, oracle.SOFTPLUS)
    np.testing.assert_allclose(ls, x, rtol=0, atol=1e-13)


def test_bounded_decay_range_and_tile_bound():
    """log g in [b, 0]; the 16-token tile cumsum never drops below 16*b
    (sec. 3.2: the reciprocal inside any 16-token tile stays in a safe range)."""
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(4096) * 8, np.full(64, 60.0), np.full(64, -60.0)])
    lam = oracle.log_decay(a, -5.0, oracle.BOUNDED)
    assert np.all(lam <= 0.0) and np.all(lam >= -5.0)
    tiles = np.cumsum(lam[: len(lam) // 16 * 16].reshape(-1, 16), axis=1)
    assert tiles.min() >= 16 * -5.0
    assert np.all(np.diff(tiles, axis=1) <= 0.0)
    # e^{-Gamma} within a tile stays finite in fp32 (e^80 < FLT_MAX)
    assert np.all(np.isfinite(np.exp(-tiles.astype(np.float32))))


def test_unbounded_decay_overflows_the_reciprocal():
    """The premise of sec. 3.1: with -softplus the tile reciprocal e^{-Gamma}
    can overflow; larger tiles raise the risk."""
    lam = oracle.log_decay(np.full(16, 10.0), -5.0, oracle.SOFTPLUS)
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.exp(-np.cumsum(lam).astype(np.float32))[-1])
    rng = np.random.default_rng(1)
    a = rng.standard_normal(1 << 16) * 2.0 + 2.0        # the ablation's logits
    lam = oracle.log_decay(a, -5.0, oracle.SOFTPLUS)
    g64 = np.cumsum(lam.reshape(-1, 64), axis=1).astype(np.float32)
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp(-g64)))


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))
    b = g["b"]
    q = np.array(g["q"]).reshape(2, 1, 1)
    k = np.array(g["k"]).reshape(2, 1, 1)
    v = np.array(g["v"]).reshape(2, 1, 1)
    a = np.array(g["a"]).reshape(2, 1)
    h0 = np.array(g["h0"]).reshape(1, 1, 1, 1)
    dO = np.array(g["dO"]).reshape(2, 1, 1)
    o, hT = oracle.fwd(q, k, v, a, b, oracle.BOUNDED, h0=h0)
    np.testing.assert_allclose(o.ravel(), g["o"], rtol=1e-14)
    np.testing.assert_allclose(hT.ravel(), [g["hT"]], rtol=1e-14)
    dq, dk, dv, da, dh0 = oracle.bwd(q, k, v, a, dO, b, oracle.BOUNDED, h0=h0)
    np.testing.assert_allclose(dq.ravel(), g["dq"], rtol=1e-14)
    np.testing.assert_allclose(dk.ravel(), g["dk"], rtol=1e-14)
    np.testing.assert_allclose(dv.ravel(), g["dv"], rtol=1e-14)
    np.testing.assert_allclose(da.ravel(), np.array(g["dlambda"]) * b / 4.0, rtol=1e-14)
    np.testing.assert_allclose(dh0.ravel(), [g["dh0"]], rtol=1e-14)


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_forward_equals_brute_force(mode):
    rng = np.random.default_rng(2 + mode)
    q, k, v, a, cu, h0 = _rand_case(rng, 70, 3, 5, 4, docs=[0, 17, 17, 50, 70])
    o, hT = oracle.fwd(q, k, v, a, -5.0, mode, h0=h0, cu_seqlens=cu)
    ob, hb = _brute_force(q, k, v, a, cu, h0, -5.0, mode)
    np.testing.assert_allclose(o, ob, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, hb, rtol=1e-11, atol=1e-12)


def test_b_zero_is_plain_causal_linear_attention():
    rng = np.random.default_rng(4)
    q, k, v, a, cu, h0 = _rand_case(rng, 40, 2, 6, 3)
    o, hT = oracle.fwd(q, k, v, a, 0.0, oracle.BOUNDED, h0=h0)
    # running sum of outer products, no decay
    kv = np.einsum("thi,thj->thij", k, v).cumsum(axis=0) + h0[0][None]
    np.testing.assert_allclose(o, np.einsum("thi,thij->thj", q, kv), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT[0], kv[-1], rtol=1e-12, atol=1e-12)
    dO = rng.standard_normal(v.shape)
    *_, da, _ = oracle.bwd(q, k, v, a, dO, 0.0, oracle.BOUNDED, h0=h0)
    assert np.all(da == 0.0)
    # continuity as b -> 0-
    o2, _ = oracle.fwd(q, k, v, a, -1e-9, oracle.BOUNDED, h0=h0)
    np.testing.assert_allclose(o2, o, rtol=1e-6, atol=1e-7)


def test_constant_decay_retention_closed_form():
    """a >= 40 gives sigmoid(a) == 1 in fp64, so log g = b for every token:
    o = (D * Q K^T) V with D_ts = e^{b (t - s)} for s <= t."""
    rng = np.random.default_rng(5)
    T, dk, dv, b = 33, 4, 3, -0.7
    q, k, v, _, _, _ = _rand_case(rng, T, 1, dk, dv, h0=False)
    a = np.full((T, 1), 40.0)
    o, _ = oracle.fwd(q, k, v, a, b, oracle.BOUNDED)
    t = np.arange(T)
    D = np.where(t[:, None] >= t[None, :], np.exp(b * (t[:, None] - t[None, :])), 0.0)
    np.testing.assert_allclose(o[:, 0], (D * (q[:, 0] @ k[:, 0].T)) @ v[:, 0], rtol=1e-12)


def test_varlen_is_concatenation_of_documents():
    rng = np.random.default_rng(6)
    docs = [0, 9, 30, 31, 64]
    q, k, v, a, cu, h0 = _rand_case(rng, 64, 2, 4, 5, docs=docs)
    o, hT = oracle.fwd(q, k, v, a, -5.0, oracle.BOUNDED, h0=h0, cu_seqlens=cu)
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(hT.shape)
    g = oracle.bwd(q, k, v, a, dO, -5.0, oracle.BOUNDED, h0=h0, dhT=dhT, cu_seqlens=cu)
    for n in range(len(docs) - 1):
        s = slice(docs[n], docs[n + 1])
        on, hn = oracle.fwd(q[s], k[s], v[s], a[s], -5.0, oracle.BOUNDED, h0=h0[n:n + 1])
        assert np.array_equal(on, o[s]) and np.array_equal(hn[0], hT[n])
        gn = oracle.bwd(q[s], k[s], v[s], a[s], dO[s], -5.0, oracle.BOUNDED, h0=h0[n:n + 1],
                        dhT=dhT[n:n + 1])
        for x, y in zip(gn[:4], g[:4]):
            assert np.array_equal(x, y[s])
        assert np.array_equal(gn[4][0], g[4][n])


def test_linearity_in_v_and_h0():
    rng = np.random.default_rng(7)
    q, k, v1, a, cu, h1 = _rand_case(rng, 30, 2, 4, 3)
    v2 = rng.standard_normal(v1.shape)
    h2 = rng.standard_normal(h1.shape)
    o1, s1 = oracle.fwd(q, k, v1, a, h0=h1)
    o2, s2 = oracle.fwd(q, k, v2, a, h0=h2)
    o3, s3 = oracle.fwd(q, k, 2 * v1 - 3 * v2, a, h0=2 * h1 - 3 * h2)
    np.testing.assert_allclose(o3, 2 * o1 - 3 * o2, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(s3, 2 * s1 - 3 * s2, rtol=1e-11, atol=1e-11)


def _loss(q, k, v, a, h0, dO, dhT, b, mode, cu):
    o, hT = oracle.fwd(q, k, v, a, b, mode, h0=h0, cu_seqlens=cu)
    return float(np.sum(o * dO) + np.sum(hT * dhT))


@pytest.mark.parametrize("mode", [oracle.BOUNDED, oracle.SOFTPLUS])
def test_gradients_match_central_finite_differences(mode):
    rng = np.random.default_rng(8 + mode)
    q, k, v, a, cu, h0 = _rand_case(rng, 37, 2, 4, 3, docs=[0, 20, 37])
    dO = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    grads = oracle.bwd(q, k, v, a, dO, -5.0, mode, h0=h0, dhT=dhT, cu_seqlens=cu, window=7)
    args = dict(q=q, k=k, v=v, a=a, h0=h0)
    names = ["q", "k", "v", "a", "h0"]
    eps = 1e-6
    for name, g in zip(names, grads):
        x = args[name]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(**args, dO=dO, dhT=dhT, b=-5.0, mode=mode, cu=cu)
            x[idx] = old - eps
            lm = _loss(**args, dO=dO, dhT=dhT, b=-5.0, mode=mode, cu=cu)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(fd - g) / np.linalg.norm(g)
        assert err < 1e-7, (name, err)


def test_backward_checkpoint_window_is_exact():
    rng = np.random.default_rng(10)
    q, k, v, a, cu, h0 = _rand_case(rng, 50, 2, 3, 4)
    dO = rng.standard_normal(v.shape)
    ref = oracle.bwd(q, k, v, a, dO, h0=h0, window=1024)
    for w in (1, 3, 16):
        got = oracle.bwd(q, k, v, a, dO, h0=h0, window=w)
        for x, y in zip(got, ref):
            assert np.array_equal(x, y)


def test_empty_document_passes_state_through():
    rng = np.random.default_rng(11)
    q, k, v, a, cu, h0 = _rand_case(rng, 10, 1, 2, 2, docs=[0, 0, 10, 10])
    o, hT = oracle.fwd(q, k, v, a, h0=h0, cu_seqlens=cu)
    assert np.array_equal(hT[0], h0[0]) and np.array_equal(hT[2], h0[2])
    dhT = rng.standard_normal(hT.shape)
    *_, dh0 = oracle.bwd(q, k, v, a, np.zeros_like(v), h0=h0, dhT=dhT, cu_seqlens=cu)
    assert np.array_equal(dh0[0], dhT[0]) and np.array_equal(dh0[2], dhT[2])
