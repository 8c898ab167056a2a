"""The bounded waits of the tensor-core kernels, exercised the way the pages'
own method never needs: a test hook makes one role of one kernel (the TMA
producer warp, the MMA warp or the epilogue warps) wait on a barrier that
nothing arrives at.  The wait runs out after a short limit; the kernel must
record BDLA_ERR_TIMEOUT in the call's status word, let its own copies and
MMAs finish, free tensor memory and return, so that the next ordinary call
on the same CUDA context still matches the fp64 oracle."""
import dataclasses

import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import compare_all, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

CASES = [(k, r) for k in ("fwd", "bwd", "seg") for r in ("producer", "mma", "epilogue")]
KERNEL = {"fwd": bdla.KERNEL_FWD, "bwd": bdla.KERNEL_BWD, "seg": bdla.KERNEL_SEG}
ROLE = {"producer": bdla.STALL_PRODUCER, "mma": bdla.STALL_MMA, "epilogue": bdla.STALL_EPILOGUE}


def _inputs():
    w = small_variant(WORKLOADS["varlen64k"], T=900, H=2, n_docs=3)
    return w, make_inputs(w, with_grad=True)


@pytest.mark.parametrize("kernel,role", CASES, ids=[f"{k}-{r}" for k, r in CASES])
def test_expired_wait_reports_timeout_and_the_context_stays_usable(kernel, role):
    w, inp = _inputs()
    g = to_device(inp)
    ws_f = bdla.Workspace(256, "cuda")
    ws_b = bdla.Workspace(256, "cuda")
    try:
        # segments of two blocks, so the segment-summary kernel runs (and its
        # CTAs see a second block) in the forward and the backward
        bdla.set_seq_split(2 if kernel == "seg" else -1)
        bdla.set_wait_limit_ns(20_000_000)
        bdla.set_test_stall(KERNEL[kernel], ROLE[role])
        o, hT, ck = bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                             ckpt_stride=128, ckpt_dtype=torch.bfloat16, ws=ws_f)
        if kernel != "fwd":
            bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                     ckpt=ck, ckpt_stride=128, ws=ws_b)
        torch.cuda.synchronize()
        st_f, st_b = ws_f.read_device_status(), ws_b.read_device_status()
    finally:
        bdla.set_test_stall(KERNEL[kernel], bdla.STALL_NONE)
        bdla.set_wait_limit_ns(0)
        bdla.set_seq_split(0)
    if kernel == "fwd":
        assert st_f == bdla.ERR_TIMEOUT
    elif kernel == "bwd":
        assert (st_f, st_b) == (bdla.OK, bdla.ERR_TIMEOUT)
    else:
        assert st_f == bdla.ERR_TIMEOUT and st_b == bdla.ERR_TIMEOUT
    # the same context runs an ordinary forward and backward to the parity bar
    gpu = run_gpu(to_device(inp), w.b, w.mode)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))
