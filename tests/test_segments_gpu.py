"""GPU parity of sequence segments (documents cut into segments, the state
and the adjoint state entering each segment found by a summary GEMM pass and
a scan over segments).  Every case forces a short segment length so that
documents span several segments with a ragged last one, and compares all
outputs with the fp64 oracle on the same bytes."""
import dataclasses

import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import compare_all, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture
def split():
    """Sets the segment length (in 128-token blocks) for one test."""
    def _set(blocks):
        bdla.set_seq_split(blocks)
    yield _set
    bdla.set_seq_split(0)


def _case(name, T, H=2, n_docs=None, **kw):
    w = small_variant(WORKLOADS[name], T=T, H=H, n_docs=n_docs)
    return dataclasses.replace(w, **kw) if kw else w


def _dhT(inp, H, dk, dv, seed=7):
    n_seq = (inp["cu_seqlens"].numel() - 1) if inp["cu_seqlens"] is not None else inp["q"].shape[0]
    return torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(seed)) * 0.1


@pytest.mark.parametrize("mode", [bdla.BOUNDED, bdla.SOFTPLUS])
@pytest.mark.parametrize("blocks", [1, 3])
def test_fixed_length_documents_across_segments(split, mode, blocks):
    kw = dict(h0_std=0.2, mode=mode, fwd_only=False)
    if mode == bdla.SOFTPLUS:
        kw.update(a_mean=2.0, a_std=2.0)
    w = dataclasses.replace(_case("c8k", 1500, **kw), B=2)
    split(blocks)
    inp = make_inputs(w, with_grad=True)
    dhT = _dhT(inp, w.H, w.dk, w.dv)
    gpu = run_gpu(to_device(inp), w.b, mode, dhT=dhT.cuda())
    compare_all(gpu, run_oracle(inp, w.b, mode, dhT=dhT))


def test_varlen_documents_shorter_and_longer_than_a_segment(split):
    w = _case("varlen64k", 1500, n_docs=3)
    inp = make_inputs(w, with_grad=True)
    inp["cu_seqlens"] = torch.tensor([0, 0, 37, 37, 700, 1300, 1300, 1500], dtype=torch.int32)
    inp["h0"] = torch.randn((7, 2, 128, 128), generator=torch.Generator().manual_seed(3)) * 0.1
    dhT = _dhT(inp, w.H, w.dk, w.dv)
    split(2)
    gpu = run_gpu(to_device(inp), w.b, w.mode, dhT=dhT.cuda())
    compare_all(gpu, run_oracle(inp, w.b, w.mode, dhT=dhT))


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 256)])
def test_head_widths_across_segments(split, dk, dv):
    w = dataclasses.replace(_case("c256k", 900, dk=dk, dv=dv, h0_std=0.1), B=1)
    split(2)
    inp = make_inputs(w, with_grad=True)
    gpu = run_gpu(to_device(inp), w.b, w.mode)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))


@pytest.mark.parametrize("stride,dtype", [(128, torch.bfloat16), (256, torch.float32),
                                          (16, torch.float32)])
def test_checkpoints_written_by_segments_feed_the_backward(split, stride, dtype):
    """Checkpoints keep their document-wide slot numbering when segments
    write them; the backward reads them (stride dividing 128) or recomputes
    the states with segments of its own (stride 256)."""
    w = _case("varlen64k", 1100, n_docs=2, h0_std=0.1)
    split(2)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    ws = bdla.Workspace(256, "cuda")
    o, hT, ck = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                         ckpt_stride=stride, ckpt_dtype=dtype, ws=ws)
    dq, dk, dv, da, dh0 = bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"],
                                   cu_seqlens=g["cu_seqlens"], ckpt=ck, ckpt_stride=stride,
                                   want_dh0=True, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
    gpu = dict(o=o, hT=hT, dq=dq, dk=dk, dv=dv, da=da, dh0=dh0)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))
    # the same checkpoints as a single CTA per document writes
    split(-1)
    _, _, ck1 = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                         ckpt_stride=stride, ckpt_dtype=dtype, ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
    # compare the slots the forward writes: block starts at multiples of the stride
    cu = inp["cu_seqlens"].tolist()
    slots = [c0 // stride + n + c for n, (c0, c1) in enumerate(zip(cu[:-1], cu[1:]))
             for c in range((c1 - c0 + stride - 1) // stride)]
    idx = torch.tensor(slots, device=ck.device)
    got, ref = ck.index_select(1, idx).float(), ck1.index_select(1, idx).float()
    err = (got - ref).norm() / ref.norm()
    assert err < 5e-3, float(err)


def test_automatic_split_engages_for_few_units():
    """Two heads of one 3000-token document are fewer units than SMs: the
    default policy cuts the document, and the result meets the bar."""
    w = dataclasses.replace(_case("c8k", 3000, h0_std=0.1), B=1)
    bdla.set_seq_split(0)
    inp = make_inputs(w, with_grad=True)
    assert bdla.workspace_bytes(bdla.OP_FWD, tuple(inp["q"].shape), w.dv) > \
        _ws_without_split(inp, w)
    gpu = run_gpu(to_device(inp), w.b, w.mode)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))


def _ws_without_split(inp, w):
    bdla.set_seq_split(-1)
    try:
        return bdla.workspace_bytes(bdla.OP_FWD, tuple(inp["q"].shape), w.dv)
    finally:
        bdla.set_seq_split(0)
