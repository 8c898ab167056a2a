"""GPU parity of the gated delta rule path (bdla_fwd_delta / bdla_bwd_delta,
through the C ABI) against the fp64 gated-delta oracle on the same seeded
bytes.  Bar per tensor: relative L2 <= 5e-3 and max-abs <= 2e-2 * max|ref|
(o, hT, dq, dk, dv, da, dbeta, dh0)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import assert_close, cu_of, flat64, heads64, to_device

pytestmark = pytest.mark.gpu


def _delta_case(name, T, H=2, n_docs=None, **kw):
    w = small_variant(WORKLOADS[name], T=T, H=H, n_docs=n_docs)
    return dataclasses.replace(w, delta=True, vec=False, **kw)


def _run(w, inp, o_dtype=torch.bfloat16, with_grad=False, dhT=None):
    g = to_device(inp)
    ws = bdla.Workspace(256, "cuda")
    o, hT = bdla.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, h0=g.get("h0"),
                           cu_seqlens=g.get("cu_seqlens"), mode=w.mode, o_dtype=o_dtype, ws=ws)
    out = dict(o=o, hT=hT)
    if with_grad:
        dq, dk, dv, da, dbeta, dh0 = bdla.bwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], g["dO"], w.b,
                                                    h0=g.get("h0"), dhT=None if dhT is None else dhT.cuda(),
                                                    cu_seqlens=g.get("cu_seqlens"), mode=w.mode, want_dh0=True,
                                                    ws=ws)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dbeta=dbeta, dh0=dh0)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
    return out


def _oracle(inp, b, mode, heads=None, with_grad=False, dhT=None):
    q = inp["q"]
    B, T = q.shape[0], q.shape[1]
    cu = cu_of(inp, B, T)
    args = [flat64(inp[x], heads) for x in ("q", "k", "v", "a", "beta")]
    h0 = heads64(inp.get("h0"), heads)
    o, hT = oracle.fwd_delta(*args, b, mode, h0=h0, cu_seqlens=cu)
    out = dict(o=o, hT=hT)
    if with_grad:
        dhT64 = None if dhT is None else heads64(dhT, heads)
        dq, dk, dv, da, dbeta, dh0 = oracle.bwd_delta(*args, flat64(inp["dO"], heads), b, mode, h0=h0, dhT=dhT64,
                                                      cu_seqlens=cu)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dbeta=dbeta, dh0=dh0)
    return out


def _compare(gpu, ref, heads=None):
    for n, r in ref.items():
        x = gpu[n]
        if n in ("hT", "dh0"):
            x = x if heads is None else x[:, heads]
            got = x.double().cpu().numpy()
        else:
            x = x if heads is None else x[:, :, heads]
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
def test_delta_fwd_bwd_small(case, mode):
    name, T, H, nd, dk, dv = case
    kw = dict(dk=dk, dv=dv, mode=mode, fwd_only=False)
    if mode == bdla.SOFTPLUS:
        kw.update(a_mean=2.0, a_std=2.0)
    w = _delta_case(name, T, H, nd, **kw)
    inp = make_inputs(w, with_grad=True)
    n_seq = (inp["cu_seqlens"].numel() - 1) if inp["cu_seqlens"] is not None else w.B
    dhT = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(9)) * 0.1
    _compare(_run(w, inp, with_grad=True, dhT=dhT), _oracle(inp, w.b, mode, with_grad=True, dhT=dhT))


@pytest.mark.parametrize("T", [1, 15, 16, 17, 33])
def test_delta_edge_lengths(T):
    w = dataclasses.replace(_delta_case("c8k", T, H=2, dk=64, dv=64, h0_std=0.3), B=2)
    inp = make_inputs(w, with_grad=True)
    _compare(_run(w, inp, o_dtype=torch.float32, with_grad=True), _oracle(inp, w.b, w.mode, with_grad=True))


def test_delta_full_write_retrieves_the_value():
    """beta = 1 and unit keys: reading with the key just written returns its
    value (the rule's defining property), whatever came before."""
    w = _delta_case("c8k", 257, H=2, dk=128, dv=128, h0_std=0.3)
    inp = make_inputs(w, with_grad=False)
    inp["beta"] = torch.ones_like(inp["beta"])
    inp["q"] = inp["k"].clone()
    gpu = _run(w, inp, o_dtype=torch.float32)
    ref = _oracle(inp, w.b, w.mode)
    _compare(gpu, ref)
    v = inp["v"].float().numpy()
    np.testing.assert_allclose(gpu["o"].cpu().numpy(), v, rtol=0, atol=0.05)


@pytest.mark.slow
def test_delta_full_size_workload_sampled_heads():
    """The 64K stage's packed documents at full size on the GPU, forward and
    backward; the oracle checks two heads (every document, every token)."""
    w = WORKLOADS["varlen64k_delta"]
    inp = make_inputs(w, with_grad=True)
    heads = [0, 21]
    gpu = _run(w, inp, with_grad=True)
    _compare(gpu, _oracle(inp, w.b, w.mode, heads=heads, with_grad=True), heads=heads)


def test_delta_states_from_the_forward_equal_the_backwards_own():
    """The forward's hand-off of the state before every tile (states_out)
    gives bitwise the same gradients as the backward's own states pass."""
    w = _delta_case("varlen64k", 900, H=2, n_docs=3, h0_std=0.2)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    st = bdla.tile_states(g["q"], g["v"], g["cu_seqlens"])
    fo = bdla.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"], states_out=st)
    fo_plain = bdla.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"])
    own = bdla.bwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                     want_dh0=True)
    handed = bdla.bwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                        want_dh0=True, states=st)
    torch.cuda.synchronize()
    for x, y in zip(fo, fo_plain):
        assert torch.equal(x, y)
    for x, y in zip(own, handed):
        assert torch.equal(x, y)


@pytest.mark.parametrize("cu", [[0, 100, 50, 300], [0, 100, 200], [0, 500]])
def test_delta_bad_cu_seqlens_set_device_status(cu):
    """Malformed packed offsets: BDLA_ERR_DEVICE from the device-side document
    check, spans outside the tensors skipped, the context still usable."""
    w = _delta_case("varlen64k", 300, H=2, n_docs=2)
    g = to_device(make_inputs(w, with_grad=False))
    bad = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ws = bdla.Workspace(256, "cuda")
    bdla.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, cu_seqlens=bad, ws=ws)
    assert ws.read_device_status() == bdla.ERR_DEVICE
    assert ws.read_device_status() == 0          # cleared after reading
    bdla.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, cu_seqlens=bad.new_tensor([0, 300]), ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
