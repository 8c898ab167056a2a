"""GPU parity of the per-channel (vector) decay path (bdla_fwd_vec /
bdla_bwd_vec, through the C ABI) against the fp64 per-channel oracle on the
same seeded bytes.  Bar per tensor: relative L2 <= 5e-3 and max-abs <=
2e-2 * max|ref| (o, hT, dq, dk, dv, da, dh0)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import assert_close, cu_of, flat64, heads64, to_device

pytestmark = pytest.mark.gpu


def _vec_case(name, T, H=2, n_docs=None, **kw):
    w = small_variant(WORKLOADS[name], T=T, H=H, n_docs=n_docs)
    return dataclasses.replace(w, vec=True, **kw)


def _run(w, inp, with_grad=True, o_dtype=torch.bfloat16, dhT=None):
    g = to_device(inp)
    ws = bdla.Workspace(256, "cuda")
    o, hT = bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, h0=g.get("h0"), cu_seqlens=g.get("cu_seqlens"),
                         mode=w.mode, o_dtype=o_dtype, ws=ws)
    out = dict(o=o, hT=hT)
    if with_grad:
        dq, dk, dv, da, dh0 = bdla.bwd_vec(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g.get("h0"),
                                           dhT=None if dhT is None else dhT.cuda(),
                                           cu_seqlens=g.get("cu_seqlens"), mode=w.mode, want_dh0=True, ws=ws)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dh0=dh0)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
    return out


def _oracle(inp, b, mode, with_grad=True, dhT=None):
    q = inp["q"]
    B, T = q.shape[0], q.shape[1]
    cu = cu_of(inp, B, T)
    args = [flat64(inp[x]) for x in ("q", "k", "v", "a")]
    h0 = heads64(inp.get("h0"), None)
    o, hT = oracle.fwd_vec(*args, b, mode, h0=h0, cu_seqlens=cu)
    out = dict(o=o, hT=hT)
    if with_grad:
        dq, dk, dv, da, dh0 = oracle.bwd_vec(*args, flat64(inp["dO"]), b, mode, h0=h0,
                                             dhT=None if dhT is None else dhT.double().numpy(), cu_seqlens=cu)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dh0=dh0)
    return out


def _compare(gpu, ref):
    for n, r in ref.items():
        x = gpu[n]
        if n in ("hT", "dh0"):
            got = x.double().cpu().numpy()
        else:
            got = x.reshape(x.shape[0] * x.shape[1], *x.shape[2:]).double().cpu().numpy()
        assert_close(n, got, r)


CASES = [
    # name, T, H, n_docs, dk, dv
    ("c8k", 300, 2, None, 128, 128),
    ("varlen64k", 700, 2, 3, 128, 128),
    ("pr1", 333, 2, None, 64, 64),
    ("c8k", 200, 3, None, 64, 128),
    ("c8k", 150, 2, None, 128, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-T{c[1]}-dk{c[4]}-dv{c[5]}")
@pytest.mark.parametrize("mode", [bdla.BOUNDED, bdla.SOFTPLUS])
def test_vec_fwd_bwd_small(case, mode):
    name, T, H, nd, dk, dv = case
    kw = dict(dk=dk, dv=dv, mode=mode, fwd_only=False)
    if mode == bdla.SOFTPLUS:
        kw.update(a_mean=2.0, a_std=2.0)
    w = _vec_case(name, T, H, nd, **kw)
    inp = make_inputs(w, with_grad=True)
    n_seq = (inp["cu_seqlens"].numel() - 1) if inp["cu_seqlens"] is not None else w.B
    dhT = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(9)) * 0.1
    _compare(_run(w, inp, dhT=dhT), _oracle(inp, w.b, mode, dhT=dhT))


@pytest.mark.parametrize("T", [1, 15, 16, 17, 33])
def test_vec_edge_lengths(T):
    w = dataclasses.replace(_vec_case("c8k", T, H=2, dk=64, dv=64, h0_std=0.3), B=2)
    inp = make_inputs(w, with_grad=True)
    _compare(_run(w, inp, o_dtype=torch.float32), _oracle(inp, w.b, w.mode))


def test_vec_saturated_decay_reaches_the_tile_floor():
    """Logits well above 0 give lambda ~ b in every channel: the diagonal
    tile's reciprocal reaches e^{80} per channel and stays finite, and the
    gate derivative (about 6e-6 |b| here) keeps its relative accuracy.  At
    a ~ 12 the fp64 oracle's 1 - sigma(a) still has ten good digits; far
    beyond it the oracle's own cancellation would dominate the comparison."""
    w = _vec_case("c8k", 200, H=2, a_mean=12.0, a_std=0.5)
    lam = w.b / (1.0 + np.exp(-12.0 + 2.5))
    assert 16 * lam < -79.9
    inp = make_inputs(w, with_grad=True)
    _compare(_run(w, inp), _oracle(inp, w.b, w.mode))


def test_vec_with_equal_channels_matches_the_scalar_path():
    """Per-channel logits equal over the key channels reproduce the scalar
    decay kernels (the tcgen05 path) within the bar."""
    w = _vec_case("varlen64k", 500, H=2, n_docs=2)
    inp = make_inputs(w, with_grad=True)
    a_s = inp["a"][..., 0].contiguous()
    inp["a"] = a_s[..., None].expand(*a_s.shape, w.dk).contiguous()
    g = to_device(inp)
    vo, vhT = bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                           o_dtype=torch.float32)
    so, shT, _ = bdla.fwd(g["q"], g["k"], g["v"], a_s.cuda(), w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                          o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close("o", vo.cpu().numpy(), so.cpu().numpy())
    assert_close("hT", vhT.cpu().numpy(), shT.cpu().numpy())


def test_vec_states_from_the_forward_equal_the_backwards_own():
    """The forward's hand-off of the state before every tile (states_out)
    gives bitwise the same gradients as the backward's own states pass."""
    w = _vec_case("varlen64k", 900, H=2, n_docs=3, h0_std=0.2)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    st = bdla.tile_states(g["q"], g["v"], g["cu_seqlens"])
    fo = bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"], states_out=st)
    fo_plain = bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"])
    own = bdla.bwd_vec(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                     want_dh0=True)
    handed = bdla.bwd_vec(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                        want_dh0=True, states=st)
    torch.cuda.synchronize()
    for x, y in zip(fo, fo_plain):
        assert torch.equal(x, y)
    for x, y in zip(own, handed):
        assert torch.equal(x, y)


@pytest.mark.parametrize("cu", [[0, 100, 50, 300], [0, 100, 200], [0, 500]])
def test_vec_bad_cu_seqlens_set_device_status(cu):
    """Malformed packed offsets (a negative length, offsets that stop short of
    the tensors, a document past their end): the call reports BDLA_ERR_DEVICE
    from the device-side document check, the kernels skip spans outside the
    tensors, and the context stays usable."""
    w = _vec_case("varlen64k", 300, H=2, n_docs=2)
    g = to_device(make_inputs(w, with_grad=False))
    bad = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ws = bdla.Workspace(256, "cuda")
    bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, cu_seqlens=bad, ws=ws)
    assert ws.read_device_status() == bdla.ERR_DEVICE
    assert ws.read_device_status() == 0          # cleared after reading
    bdla.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, cu_seqlens=bad.new_tensor([0, 300]), ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
