"""GPU parity of the recurrent decode step (one token per sequence against a
resident fp32 state) with the fp64 oracle's token-by-token recurrence: single
steps, several steps in a row, and a chunked prefill handing its final state
over to decode steps."""
import numpy as np
import pytest
import torch

import oracle
from chunked_linear_attention_bounded_gb300 import bdla

from _parity import assert_close

pytestmark = pytest.mark.gpu


def _tokens(n_seq, H, dk, dv, steps, seed, a_mean=0.0, a_std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((steps, n_seq, H, dk), generator=g) / dk ** 0.5).bfloat16()
    k = torch.randn((steps, n_seq, H, dk), generator=g)
    k = (k / k.norm(dim=-1, keepdim=True)).bfloat16()
    v = torch.randn((steps, n_seq, H, dv), generator=g).bfloat16()
    a = torch.randn((steps, n_seq, H), generator=g) * a_std + a_mean
    return q, k, v, a


def _oracle_steps(q, k, v, a, h0, b, mode):
    """The oracle on each sequence's `steps` tokens from h0: o [steps, N, H, dv], hT."""
    steps, n_seq, H = a.shape
    # sequence-major packing: sequence n owns tokens n*steps .. n*steps+steps-1
    pk = lambda t: t.double().transpose(0, 1).reshape(n_seq * steps, *t.shape[2:]).numpy()
    cu = np.arange(n_seq + 1, dtype=np.int64) * steps
    o, hT = oracle.fwd(pk(q), pk(k), pk(v), pk(a), b, mode, h0=h0.double().numpy(), cu_seqlens=cu)
    o = o.reshape(n_seq, steps, H, -1).transpose(1, 0, 2, 3)
    return o, hT


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 256)])
@pytest.mark.parametrize("mode", [bdla.BOUNDED, bdla.SOFTPLUS])
def test_decode_steps_match_the_recurrence(dk, dv, mode):
    n_seq, H, steps = 5, 3, 4
    q, k, v, a = _tokens(n_seq, H, dk, dv, steps, seed=21, a_mean=2.0 if mode else 0.0)
    h0 = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(22)) * 0.2
    ref_o, ref_hT = _oracle_steps(q, k, v, a, h0, -5.0, mode)
    state = h0.clone().cuda()
    for t in range(steps):
        o = bdla.decode(q[t].cuda(), k[t].cuda(), v[t].cuda(), a[t].cuda(), state, b=-5.0, mode=mode,
                        o_dtype=torch.float32)
        torch.cuda.synchronize()
        assert_close(f"o[{t}]", o.cpu().numpy(), ref_o[t])
    assert_close("state", state.cpu().numpy(), ref_hT)


def test_decode_bf16_output():
    n_seq, H, dk, dv = 7, 2, 128, 128
    q, k, v, a = _tokens(n_seq, H, dk, dv, 1, seed=23)
    h0 = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(24)) * 0.2
    ref_o, ref_hT = _oracle_steps(q, k, v, a, h0, -5.0, bdla.BOUNDED)
    state = h0.clone().cuda()
    o = bdla.decode(q[0].cuda(), k[0].cuda(), v[0].cuda(), a[0].cuda(), state)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16
    assert_close("o", o.float().cpu().numpy(), ref_o[0])
    assert_close("state", state.cpu().numpy(), ref_hT)


def test_chunked_prefill_hands_over_to_decode():
    """Forward over a prompt (tensor-core chunked path), then decode steps from
    its hT: the same outputs and final state as the recurrence over the whole
    sequence."""
    n_seq, H, dk, dv, L, steps = 2, 2, 128, 128, 300, 3
    q, k, v, a = _tokens(n_seq, H, dk, dv, L + steps, seed=25)
    h0 = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(26)) * 0.1
    ref_o, ref_hT = _oracle_steps(q, k, v, a, h0, -5.0, bdla.BOUNDED)
    bt = lambda x: x[:L].transpose(0, 1).contiguous().cuda()   # [B, T, H, d]
    o_pre, hT, _ = bdla.fwd(bt(q), bt(k), bt(v), bt(a), -5.0, h0=h0.cuda(), o_dtype=torch.float32)
    state = hT
    outs = []
    for t in range(L, L + steps):
        outs.append(bdla.decode(q[t].cuda(), k[t].cuda(), v[t].cuda(), a[t].cuda(), state,
                                o_dtype=torch.float32).cpu().numpy())
    torch.cuda.synchronize()
    assert_close("prefill o", o_pre.transpose(0, 1).cpu().numpy(), ref_o[:L])
    for i, t in enumerate(range(L, L + steps)):
        assert_close(f"decode o[{t}]", outs[i], ref_o[t])
    assert_close("state", state.cpu().numpy(), ref_hT)
