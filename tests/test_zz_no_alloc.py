"""bdla_fwd_noalloc: the forward entry point for callers that cannot allocate
device memory (for example code running inside an allocator's callbacks, or
a runtime that only provides fixed buffers for inputs and outputs).  Its
scratch is a fixed array inside the library, so these tests check that two
calls in a row, on different inputs, each match the ordinary bdla_fwd (which
takes a caller workspace) within the parity tolerance, and that a problem
larger than the fixed scratch is refused before any launch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone and after the other tests."""
import ctypes
import dataclasses

import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import assert_close, to_device

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(g, w, o, hT):
    B, T, H, dk = g["q"].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return bdla.lib().bdla_fwd_noalloc(
        _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]), _ptr(g["a"]), w.b, 16, _ptr(g["h0"]), _ptr(o),
        1 if o.dtype == torch.float32 else 0, _ptr(hT), bdla.Dims(B, T, H, dk, g["v"].shape[-1]),
        w.mode, stream)


def test_noalloc_forward_matches_bdla_fwd_on_two_calls_in_a_row():
    cases = [(128, torch.bfloat16, bdla.BOUNDED), (64, torch.float32, bdla.BOUNDED)]
    for i, (dv, odt, mode) in enumerate(cases):
        w = small_variant(WORKLOADS["c8k"], T=700, H=3, seed_offset=40 + i)
        w = dataclasses.replace(w, dv=dv, h0_std=0.2, mode=mode)
        g = to_device(make_inputs(w, with_grad=False))
        ref_o, ref_hT, _ = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], mode=mode,
                                    o_dtype=odt)
        o = torch.full_like(ref_o, float("nan"))
        hT = torch.full_like(ref_hT, float("nan"))
        assert _call_noalloc(g, w, o, hT) == 0
        torch.cuda.synchronize()
        assert_close(f"o[call {i}]", o.float().cpu().numpy(), ref_o.float().cpu().numpy())
        assert_close(f"hT[call {i}]", hT.cpu().numpy(), ref_hT.cpu().numpy())


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 2^21 (token, head) pairs is the limit; every pointer below is rejected
    # by the host-side size check before any launch.
    fake = ctypes.c_void_p(1 << 20)
    dims = bdla.Dims(1, (1 << 21) // 4 + 16, 4, 128, 128)
    st = bdla.lib().bdla_fwd_noalloc(fake, fake, fake, fake, -5.0, 16, None, fake, 0, None, dims, 0,
                                     None)
    assert st == 10
    assert "fixed scratch" in bdla.status_string(st)
