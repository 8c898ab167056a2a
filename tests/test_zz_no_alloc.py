"""bdla_fwd_noalloc: the forward entry point for callers that cannot allocate
device memory (for example code running inside an allocator's callbacks, or
a runtime that only provides fixed buffers for inputs and outputs).  Its
only scratch is a status word inside the library, so these tests check that
two calls in a row, on different inputs, each match the ordinary bdla_fwd
(which takes a caller workspace) and the fp64 oracle within the parity
tolerance, that each call leaves no device-side error in the library's status
word (read through bdla_noalloc_read_status), and that problems beyond the
token coordinates or the grid limits are refused before any launch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone and after the other tests."""
import ctypes
import dataclasses

import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import assert_close, gpu_to_ref_layout, run_oracle, to_device


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(g, w, o, hT):
    B, T, H, dk = g["q"].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return bdla.lib().bdla_fwd_noalloc(
        _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]), _ptr(g["a"]), w.b, 16, _ptr(g["h0"]), _ptr(o),
        1 if o.dtype == torch.float32 else 0, _ptr(hT), bdla.Dims(B, T, H, dk, g["v"].shape[-1]),
        w.mode, stream)


def _read_noalloc_status():
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return bdla.lib().bdla_noalloc_read_status(stream)


@pytest.mark.gpu
def test_noalloc_forward_matches_bdla_fwd_and_oracle_on_two_calls_in_a_row():
    cases = [(128, torch.bfloat16, bdla.BOUNDED), (64, torch.float32, bdla.SOFTPLUS)]
    for i, (dv, odt, mode) in enumerate(cases):
        w = small_variant(WORKLOADS["c8k"], T=700, H=3, seed_offset=40 + i)
        w = dataclasses.replace(w, dv=dv, h0_std=0.2, mode=mode)
        if mode == bdla.SOFTPLUS:
            w = dataclasses.replace(w, a_mean=2.0, a_std=2.0)
        inp = make_inputs(w, with_grad=False)
        g = to_device(inp)
        ref_o, ref_hT, _ = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], mode=mode,
                                    o_dtype=odt)
        o = torch.full_like(ref_o, float("nan"))
        hT = torch.full_like(ref_hT, float("nan"))
        assert _call_noalloc(g, w, o, hT) == bdla.OK
        assert _read_noalloc_status() == bdla.OK, f"call {i} recorded a device-side error"
        # against the entry point that takes a workspace
        assert_close(f"o[call {i}] vs bdla_fwd", o.float().cpu().numpy(), ref_o.float().cpu().numpy())
        assert_close(f"hT[call {i}] vs bdla_fwd", hT.cpu().numpy(), ref_hT.cpu().numpy())
        # against the fp64 oracle
        ref = run_oracle(inp, w.b, mode, with_grad=False)
        assert_close(f"o[call {i}] vs oracle", gpu_to_ref_layout("o", o.float()), ref["o"])
        assert_close(f"hT[call {i}] vs oracle", gpu_to_ref_layout("hT", hT), ref["hT"])


def test_noalloc_refuses_problems_beyond_its_token_coordinates_or_the_grid():
    # Every pointer below is fake and never dereferenced: each call is
    # rejected by a host-side check before any launch (no GPU needed).
    fake = ctypes.c_void_p(1 << 20)
    L = bdla.lib()

    def call(dims):
        return L.bdla_fwd_noalloc(fake, fake, fake, fake, -5.0, 16, None, fake, 0, None, dims, 0, None)

    # B * T = 2^31 tokens is one more than the 32-bit token coordinates address
    st = call(bdla.Dims(2, 1 << 30, 1, 128, 128))
    assert st == bdla.ERR_TOO_LARGE
    assert "2^31 - 1" in bdla.status_string(st)
    # B * T * H = 2^15 * 2^30 * 2^19 wraps to 0 in 64-bit arithmetic; refused all the same
    assert call(bdla.Dims(1 << 15, 1 << 30, 1 << 19, 128, 128)) == bdla.ERR_TOO_LARGE
    assert call(bdla.Dims(1 << 15, (1 << 31) - 1, 1 << 19, 128, 128)) == bdla.ERR_TOO_LARGE
    # more documents than a grid extent holds
    assert call(bdla.Dims(65536, 1, 1, 64, 64)) == bdla.ERR_UNSUPPORTED
    assert call(bdla.Dims(1, 64, 2, 256, 64)) == bdla.ERR_UNSUPPORTED
