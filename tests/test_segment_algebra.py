"""fp64 restatement of the segment scan the kernels use when a document is cut
into segments (summary, scan, rerun), checked against the token-by-token
oracle.  It pins the algebra of that evaluation order, not the kernels.

The pages say only that a recurrent state passes between chunks
("Engineering Long-Context Training for Trillion-Parameter MoE Models",
sec. 3.1); the reading taken here: with Lam_t the inclusive cumulative
log-decay from the segment start,
  state summary    U_s = sum_t e^{Lam_end - Lam_t} k_t v_t^T     (suffix weights <= 1)
  adjoint summary  R_s = sum_t e^{Lam_t} q_t dO_t^T              (prefix weights <= 1)
  scan             S_in(s+1) = e^{Lam_end(s)} S_in(s) + U_s,      S_in(0) = h0
                   D_in(s)   = e^{Lam_end(s)} D_in(s+1) + R_s,    D_in(n) = dhT
and every segment is then run on its own from S_in(s) with the adjoint
D_in(s+1) arriving at its end.
"""
import numpy as np
import pytest

import oracle


def _segments(L, seg):
    return [(s, min(s + seg, L)) for s in range(0, L, seg)]


def summaries(q, k, v, dO, lam, seg, suffix_state=True):
    """Per segment: (U, R, Lam_end) for one head; q,k [L,dk], v,dO [L,dv], lam [L]."""
    out = []
    for s, e in _segments(len(lam), seg):
        Lam = np.cumsum(lam[s:e])
        Lend = Lam[-1]
        ws = np.exp(Lend - Lam) if suffix_state else np.exp(Lam)
        U = (k[s:e] * ws[:, None]).T @ v[s:e]
        R = (q[s:e] * np.exp(Lam)[:, None]).T @ dO[s:e]
        out.append((U, R, Lend))
    return out


def segmented_run(q, k, v, a, dO, b, mode, h0, dhT, seg, suffix_state=True):
    """o, hT, dq, dk, dv, da, dh0 of one document and one head from per-segment
    oracle runs joined by the summary scan."""
    lam = oracle.log_decay(a, b, mode)
    sm = summaries(q, k, v, dO, lam, seg, suffix_state)
    spans = _segments(len(a), seg)
    S_in = [h0]
    for U, _, Lend in sm:
        S_in.append(np.exp(Lend) * S_in[-1] + U)
    D_in = [None] * len(sm) + [dhT]
    for i in reversed(range(len(sm))):
        _, R, Lend = sm[i]
        D_in[i] = np.exp(Lend) * D_in[i + 1] + R
    o = np.zeros_like(v)
    grads = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(a)]
    for i, (s, e) in enumerate(spans):
        x = lambda t: t[s:e, None]
        oi, _ = oracle.fwd(x(q), x(k), x(v), x(a), b, mode, h0=S_in[i][None, None])
        o[s:e] = oi[:, 0]
        gi = oracle.bwd(x(q), x(k), x(v), x(a), x(dO), b, mode, h0=S_in[i][None, None],
                        dhT=D_in[i + 1][None, None])
        for acc, g in zip(grads, gi[:4]):
            acc[s:e] = g[:, 0]
    return o, S_in[-1], grads, D_in[0]


def _case(rng, L, dk, dv, mode):
    q = rng.standard_normal((L, dk)) * 0.4
    k = rng.standard_normal((L, dk)) * 0.4
    v = rng.standard_normal((L, dv))
    dO = rng.standard_normal((L, dv))
    a = rng.standard_normal(L) * 2.0 + (2.0 if mode == oracle.SOFTPLUS else 0.0)
    h0 = rng.standard_normal((dk, dv)) * 0.3
    dhT = rng.standard_normal((dk, dv)) * 0.3
    return q, k, v, a, dO, h0, dhT


@pytest.mark.parametrize("mode,L,seg", [(oracle.BOUNDED, 300, 64), (oracle.BOUNDED, 128, 128),
                                        (oracle.SOFTPLUS, 200, 48), (oracle.BOUNDED, 45, 16),
                                        (oracle.BOUNDED, 257, 128)])
def test_segment_scan_equals_the_whole_document(mode, L, seg):
    rng = np.random.default_rng(L + 7 * seg + mode)
    dk, dv, b = 6, 5, -5.0
    q, k, v, a, dO, h0, dhT = _case(rng, L, dk, dv, mode)
    o, hT, (dq, dk_, dv_, da), dh0 = segmented_run(q, k, v, a, dO, b, mode, h0, dhT, seg)
    ro, rhT = oracle.fwd(q[:, None], k[:, None], v[:, None], a[:, None], b, mode, h0=h0[None, None])
    rq, rk, rv, rda, rdh0 = oracle.bwd(q[:, None], k[:, None], v[:, None], a[:, None], dO[:, None], b, mode,
                                       h0=h0[None, None], dhT=dhT[None, None])
    for got, ref in ((o, ro[:, 0]), (hT, rhT[0, 0]), (dq, rq[:, 0]), (dk_, rk[:, 0]), (dv_, rv[:, 0]),
                     (da, rda[:, 0]), (dh0, rdh0[0, 0])):
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-10)


def test_summary_weights_never_exceed_one():
    """Suffix and prefix weights are products of per-token decays <= 1, so a
    segment of any length sums without overflow (unlike a reciprocal)."""
    rng = np.random.default_rng(3)
    for mode in (oracle.BOUNDED, oracle.SOFTPLUS):
        lam = oracle.log_decay(rng.standard_normal(4096) * 3.0, -5.0, mode)
        Lam = np.cumsum(lam)
        assert np.all(Lam <= 0.0) and np.all(Lam[-1] - Lam <= 0.0)


def test_prefix_weights_for_the_state_summary_are_wrong():
    """The state summary needs the suffix weights e^{Lam_end - Lam_t}: with the
    prefix weights the joined segments no longer match the whole document."""
    rng = np.random.default_rng(11)
    q, k, v, a, dO, h0, dhT = _case(rng, 200, 6, 5, oracle.BOUNDED)
    o, hT, _, _ = segmented_run(q, k, v, a, dO, -5.0, oracle.BOUNDED, h0, dhT, 64, suffix_state=False)
    ro, rhT = oracle.fwd(q[:, None], k[:, None], v[:, None], a[:, None], -5.0, oracle.BOUNDED,
                         h0=h0[None, None])
    assert np.max(np.abs(o - ro[:, 0])) > 1e-3
    assert np.max(np.abs(hT - rhT[0, 0])) > 1e-3
