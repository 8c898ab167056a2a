"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded bytes, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from chunked_linear_attention_bounded_gb300 import bdla

# Parity bar, per tensor: relative L2 error and max-abs error relative to the
# largest reference magnitude.
REL_L2 = 5e-3
MAX_ABS = 2e-2


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def assert_close(name: str, got, ref, rel=REL_L2, max_abs=MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    e = rel_l2(got, ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    m = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert e <= rel, f"{name}: rel L2 {e:.3e} > {rel:.1e}"
    assert m <= max_abs * max(scale, 1e-30) or scale == 0.0, \
        f"{name}: max abs err {m:.3e} > {max_abs:.0e} * {scale:.3e}"
    return e


def cu_of(inp, B, T) -> np.ndarray:
    if inp.get("cu_seqlens") is not None:
        return inp["cu_seqlens"].numpy().astype(np.int64)
    return np.arange(B + 1, dtype=np.int64) * T


def flat64(t: torch.Tensor, heads=None) -> np.ndarray:
    """[B, T, H, d] (or [B, T, H]) CPU tensor -> float64 [B*T, H', d] for the oracle."""
    x = t
    if heads is not None:
        x = x[:, :, heads]
    x = x.reshape(x.shape[0] * x.shape[1], *x.shape[2:])
    return x.double().numpy()


def heads64(t, heads):
    if t is None:
        return None
    x = t if heads is None else t[:, heads]
    return x.double().numpy()


def to_device(inp, dev="cuda:0"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_oracle(inp, b, mode, heads=None, dhT=None, with_grad=True):
    q = inp["q"]
    B, T = q.shape[0], q.shape[1]
    cu = cu_of(inp, B, T)
    args = [flat64(inp[x], heads) for x in ("q", "k", "v", "a")]
    h0 = heads64(inp.get("h0"), heads)
    o, hT = oracle.fwd(*args, b, mode, h0=h0, cu_seqlens=cu)
    out = dict(o=o, hT=hT)
    if with_grad:
        dq, dk, dv, da, dh0 = oracle.bwd(*args, flat64(inp["dO"], heads), b, mode, h0=h0,
                                         dhT=heads64(dhT, heads), cu_seqlens=cu)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dh0=dh0)
    return out


def run_gpu(g, b, mode, with_grad=True, o_dtype=torch.bfloat16, dhT=None, ckpt_stride=0,
            bwd_ckpt=False):
    """Forward (and backward) through the C ABI; fails if a kernel recorded a
    device-side error (e.g. a bounded wait that expired)."""
    ws_f = bdla.Workspace(256, g["q"].device)
    ws_b = bdla.Workspace(256, g["q"].device)
    o, hT, ckpt = bdla.fwd(g["q"], g["k"], g["v"], g["a"], b, h0=g.get("h0"),
                           cu_seqlens=g.get("cu_seqlens"), mode=mode, o_dtype=o_dtype,
                           ckpt_stride=ckpt_stride, ws=ws_f)
    out = dict(o=o, hT=hT, ckpt=ckpt)
    if with_grad:
        dq, dk, dv, da, dh0 = bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], b, h0=g.get("h0"),
                                       dhT=dhT, cu_seqlens=g.get("cu_seqlens"),
                                       ckpt=ckpt if bwd_ckpt else None,
                                       ckpt_stride=ckpt_stride if bwd_ckpt else 0, mode=mode,
                                       want_dh0=True, ws=ws_b)
        out.update(dq=dq, dk=dk, dv=dv, da=da, dh0=dh0)
    torch.cuda.synchronize()
    assert ws_f.read_device_status() == 0, "forward recorded a device-side error"
    assert ws_b.read_device_status() == 0, "backward recorded a device-side error"
    return out


def gpu_to_ref_layout(name, t: torch.Tensor, heads=None) -> np.ndarray:
    if name in ("hT", "dh0"):
        x = t if heads is None else t[:, heads]
        return x.double().cpu().numpy()
    x = t if heads is None else t[:, :, heads]
    x = x.reshape(x.shape[0] * x.shape[1], *x.shape[2:])
    return x.double().cpu().numpy()


def compare_all(gpu, ref, heads=None, names=None):
    errs = {}
    for n in names or ref.keys():
        errs[n] = assert_close(n, gpu_to_ref_layout(n, gpu[n], heads), ref[n])
    return errs
