"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded bytes.  Bar per tensor: relative L2 <= 5e-3 and max-abs
<= 2e-2 * max|ref| (o, hT, dq, dk, dv, da, dh0)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, Workload, make_inputs, small_variant

from _parity import (assert_close, compare_all, cu_of, flat64, heads64, run_gpu, run_oracle,
                     to_device)

pytestmark = pytest.mark.gpu


def _small(name, T, H=2, n_docs=None, **kw):
    w = small_variant(WORKLOADS[name], T=T, H=H, n_docs=n_docs)
    return dataclasses.replace(w, **kw) if kw else w


@pytest.mark.parametrize("mode", [bdla.BOUNDED, bdla.SOFTPLUS])
def test_decay_kernel_tile_cumsum(mode):
    w = _small("varlen64k", T=777, H=3, n_docs=4, mode=mode, a_std=3.0)
    inp = make_inputs(w, with_grad=False)
    g = to_device(inp)
    gamma = bdla.decay(g["a"], w.b, cu_seqlens=g["cu_seqlens"], mode=mode).cpu().double().numpy().T
    lam = oracle.log_decay(inp["a"].double().numpy()[0], w.b, mode)
    ref = np.zeros_like(lam)
    cu = inp["cu_seqlens"].numpy()
    for n in range(len(cu) - 1):
        for c0 in range(cu[n], cu[n + 1], 16):
            c1 = min(c0 + 16, cu[n + 1])
            ref[c0:c1] = np.cumsum(lam[c0:c1], axis=0)
    np.testing.assert_allclose(gamma, ref, rtol=2e-5, atol=2e-5)
    if mode == bdla.BOUNDED:
        assert gamma.min() >= 16 * w.b - 1e-3 and gamma.max() <= 0.0


CASES = [
    # name, T, H, n_docs, dk, dv
    ("c8k", 300, 2, None, 128, 128),
    ("varlen64k", 700, 2, 3, 128, 128),
    ("c256k", 290, 2, None, 128, 256),
    ("pr1", 333, 2, None, 64, 64),
    ("c8k", 200, 3, None, 64, 128),
    ("c8k", 150, 2, None, 128, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-T{c[1]}-dk{c[4]}-dv{c[5]}")
@pytest.mark.parametrize("mode", [bdla.BOUNDED, bdla.SOFTPLUS])
def test_fwd_bwd_small(case, mode):
    name, T, H, nd, dk, dv = case
    kw = dict(dk=dk, dv=dv, mode=mode, fwd_only=False)
    if mode == bdla.SOFTPLUS:
        kw.update(a_mean=2.0, a_std=2.0)
    w = _small(name, T, H, nd, **kw)
    inp = make_inputs(w, with_grad=True)
    n_seq = (inp["cu_seqlens"].numel() - 1) if inp["cu_seqlens"] is not None else w.B
    dhT = torch.randn((n_seq, H, dk, dv), generator=torch.Generator().manual_seed(5)) * 0.1
    gpu = run_gpu(to_device(inp), w.b, mode, dhT=dhT.cuda())
    ref = run_oracle(inp, w.b, mode, dhT=dhT)
    compare_all(gpu, ref)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 33, 128, 129])
def test_edge_lengths(T):
    w = _small("c8k", T, H=2, dk=64, dv=64, h0_std=0.3)
    w = dataclasses.replace(w, B=2)
    inp = make_inputs(w, with_grad=True)
    gpu = run_gpu(to_device(inp), w.b, w.mode, o_dtype=torch.float32)
    ref = run_oracle(inp, w.b, w.mode)
    compare_all(gpu, ref)


def test_fp32_output_is_closer_than_bf16_output():
    """The 256-token parity workload asks for an fp32 o: it skips the final
    bf16 rounding of o, so its error against the oracle is below the bf16
    output's (both within the bar)."""
    w = WORKLOADS["pr1"]
    inp = make_inputs(w)
    ref = run_oracle(inp, w.b, w.mode, with_grad=False)
    e32 = compare_all(run_gpu(to_device(inp), w.b, w.mode, with_grad=False, o_dtype=torch.float32), ref)
    e16 = compare_all(run_gpu(to_device(inp), w.b, w.mode, with_grad=False, o_dtype=torch.bfloat16), ref)
    print("rel L2 of o: fp32 output %.3e, bf16 output %.3e" % (e32["o"], e16["o"]))
    assert e32["o"] < e16["o"]


def test_varlen_with_empty_documents():
    w = _small("varlen64k", 200, H=2, n_docs=3)
    inp = make_inputs(w, with_grad=True)
    inp["cu_seqlens"] = torch.tensor([0, 0, 37, 37, 150, 200, 200], dtype=torch.int32)
    inp["h0"] = torch.randn((6, 2, 128, 128), generator=torch.Generator().manual_seed(3)) * 0.1
    gpu = run_gpu(to_device(inp), w.b, w.mode)
    ref = run_oracle(inp, w.b, w.mode)
    compare_all(gpu, ref)


def test_zero_tokens_passes_state_through():
    h0 = torch.randn((2, 2, 64, 64), device="cuda")
    z = lambda *s, dt=torch.bfloat16: torch.zeros(s, dtype=dt, device="cuda")
    o, hT, _ = bdla.fwd(z(2, 0, 2, 64), z(2, 0, 2, 64), z(2, 0, 2, 64), z(2, 0, 2, dt=torch.float32),
                        h0=h0)
    torch.cuda.synchronize()
    assert torch.equal(hT, h0)


def test_checkpoints_are_prefix_states_and_feed_the_backward():
    w = _small("c256k", 200, H=2, dk=64, dv=128, h0_std=0.2)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    gpu = run_gpu(g, w.b, w.mode, ckpt_stride=16, bwd_ckpt=True)
    ck = gpu["ckpt"].cpu().double().numpy()          # [H, slots, dk, dv]
    q, k, v, a = (flat64(inp[x]) for x in ("q", "k", "v", "a"))
    h0 = heads64(inp["h0"], None)
    for c in range(0, 200 // 16 + 1):
        t = c * 16
        if t >= 200:
            break
        _, st = oracle.fwd(q[:t], k[:t], v[:t], a[:t], w.b, w.mode, h0=h0, cu_seqlens=[0, t])
        assert_close(f"ckpt[{c}]", ck[:, c], st[0])
    ref = run_oracle(inp, w.b, w.mode)
    compare_all(gpu, ref, names=("o", "hT", "dq", "dk", "dv", "da", "dh0"))


@pytest.mark.parametrize("dv", [64, 128])
def test_bf16_block_checkpoints_feed_the_backward(dv):
    """Forward hands the backward bf16 states every 128 tokens (the training
    step's path); the gradients still meet the bar."""
    w = _small("varlen64k", 900, H=2, n_docs=3, dv=dv)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    ws = bdla.Workspace(256, "cuda")
    o, hT, ck = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                         ckpt_stride=128, ckpt_dtype=torch.bfloat16, ws=ws)
    dq, dk, dv_, da, dh0 = bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"],
                                    cu_seqlens=g["cu_seqlens"], ckpt=ck, ckpt_stride=128, want_dh0=True,
                                    ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0
    gpu = dict(o=o, hT=hT, dq=dq, dk=dk, dv=dv_, da=da, dh0=dh0)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))


@pytest.mark.parametrize("stride,dv", [(16, 256), (32, 128), (64, 256)])
def test_fp32_inner_checkpoints_give_the_bf16_block_state_gradients(stride, dv):
    """fp32 checkpoints whose stride divides 128 reach the backward as bf16
    copies of their block-start states: the gradients are bitwise those of
    the forward's own bf16 block checkpoints (the same fp32 states rounded the
    same way), on packed documents of ragged lengths, and meet the oracle's
    bar.  dv = 256 runs the backward's second value slice."""
    w = _small("varlen64k", 900, H=2, n_docs=3, dv=dv, h0_std=0.2)
    inp = make_inputs(w, with_grad=True)
    g = to_device(inp)
    grads = {}
    for s, dt in ((stride, torch.float32), (128, torch.bfloat16)):
        ws = bdla.Workspace(256, "cuda")
        o, hT, ck = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                             ckpt_stride=s, ckpt_dtype=dt, ws=ws)
        grads[s] = bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"],
                            cu_seqlens=g["cu_seqlens"], ckpt=ck, ckpt_stride=s, want_dh0=True, ws=ws)
        torch.cuda.synchronize()
        assert ws.read_device_status() == 0
    for x, y in zip(grads[stride], grads[128]):
        assert torch.equal(x, y)
    dq, dk, dv_, da, dh0 = grads[stride]
    compare_all(dict(dq=dq, dk=dk, dv=dv_, da=da, dh0=dh0), run_oracle(inp, w.b, w.mode),
                names=("dq", "dk", "dv", "da", "dh0"))


@pytest.mark.parametrize("cu", [[0, 100, 50, 300], [0, 100, 200], [0, 500]])
def test_bad_cu_seqlens_set_device_status(cu):
    w = _small("varlen64k", 300, H=2, n_docs=2)
    inp = make_inputs(w, with_grad=False)
    g = to_device(inp)
    g["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ws = bdla.Workspace(1 << 20, "cuda")
    bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, cu_seqlens=g["cu_seqlens"], ws=ws)
    assert ws.read_device_status() == bdla.ERR_DEVICE
    assert ws.read_device_status() == 0          # cleared after reading
    # the context is still usable
    o, _, _ = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, cu_seqlens=g["cu_seqlens"][:1].new_tensor([0, 300]), ws=ws)
    torch.cuda.synchronize()
    assert ws.read_device_status() == 0


# Full-size workloads: the GPU runs the whole input, the oracle checks a
# sample of heads (every document of those heads, every token).
FULL = [("pr1", None), ("c8k", [0, 9]), ("varlen64k", [0, 17, 31]), ("c256k", [5, 12]),
        ("c1m", [3, 6]), ("c1m_ablation", [1, 6])]


@pytest.mark.slow
@pytest.mark.parametrize("name,heads", FULL, ids=[f[0] for f in FULL])
def test_full_size_workload(name, heads):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    g = to_device(inp)
    with_grad = not w.fwd_only
    gpu = run_gpu(g, w.b, w.mode, with_grad=with_grad,
                  o_dtype=torch.float32 if w.o_f32 else torch.bfloat16,
                  ckpt_stride=w.ckpt_stride, bwd_ckpt=bool(w.ckpt_stride))
    del g
    ref = run_oracle(inp, w.b, w.mode, heads=heads, with_grad=with_grad)
    compare_all(gpu, ref, heads=heads)
