"""GPU parity across decay regimes: the bound b (including b = 0, plain causal
linear attention), logits that saturate the sigmoid so the in-tile cumulative
decay reaches its floor 16 b = -80 (the largest e^{-Gamma} factor the bounded
fold ever applies), and unbounded logits strong or weak enough that the
ablation's in-tile reciprocal overflows or barely decays."""
import dataclasses

import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import compare_all, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _case(T=600, H=2, **kw):
    w = small_variant(WORKLOADS["varlen64k"], T=T, H=H, n_docs=3)
    return dataclasses.replace(w, **kw)


def _check(w):
    inp = make_inputs(w, with_grad=True)
    n_seq = inp["cu_seqlens"].numel() - 1
    dhT = torch.randn((n_seq, w.H, w.dk, w.dv), generator=torch.Generator().manual_seed(11)) * 0.1
    gpu = run_gpu(to_device(inp), w.b, w.mode, dhT=dhT.cuda())
    compare_all(gpu, run_oracle(inp, w.b, w.mode, dhT=dhT))


@pytest.mark.parametrize("b", [0.0, -0.5, -2.5, -5.0])
def test_bound_values(b):
    _check(_case(b=b))


@pytest.mark.parametrize("a_mean", [6.0, 12.0])
def test_saturated_bounded_decay_reaches_the_tile_floor(a_mean):
    # sigma(a) -> 1: every log-decay is close to b = -5, a 16-token tile's
    # cumulative decay reaches -80 and the diagonal fold uses e^{80}
    w = _case(a_mean=a_mean, a_std=0.5)
    inp = make_inputs(w, with_grad=False)
    lam = w.b / (1.0 + torch.exp(-inp["a"].double()))
    assert float(lam.max()) < -4.8
    _check(w)


@pytest.mark.parametrize("a_mean,a_std", [(8.0, 1.0), (-6.0, 1.0)])
def test_unbounded_ablation_extremes(a_mean, a_std):
    # strong decay (about -8 per token: e^{-Gamma} would pass e^{128} inside a
    # tile) and weak decay (about -0.0025 per token)
    _check(_case(mode=bdla.SOFTPLUS, a_mean=a_mean, a_std=a_std))


def test_half_width_heads_with_initial_states_and_no_segments():
    bdla.set_seq_split(-1)
    try:
        w = _case(T=700, H=3, dk=64, dv=64, h0_std=0.3)
        _check(w)
    finally:
        bdla.set_seq_split(0)
