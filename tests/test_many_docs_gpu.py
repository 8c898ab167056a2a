"""GPU parity with many packed documents: hundreds of short documents (the
longest-first document order), more documents than the order kernel ranks
(index order), and many documents cut into segments (the slot search over
the document offsets)."""
import numpy as np
import pytest
import torch

from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant

from _parity import compare_all, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _packed(lengths, H, dk, dv, seed):
    lengths = np.asarray(lengths, dtype=np.int64)
    T = int(lengths.sum())
    w = small_variant(WORKLOADS["varlen64k"], T=T, H=H, n_docs=2)
    import dataclasses
    w = dataclasses.replace(w, dk=dk, dv=dv, seed=seed)
    inp = make_inputs(w, with_grad=True)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    inp["cu_seqlens"] = torch.from_numpy(cu)
    n = len(lengths)
    inp["h0"] = torch.randn((n, H, dk, dv), generator=torch.Generator().manual_seed(seed)) * 0.1
    return w, inp


@pytest.mark.parametrize("n_docs,max_len,H", [(300, 40, 2), (4500, 6, 1)])
def test_many_short_documents(n_docs, max_len, H):
    rng = np.random.default_rng(n_docs)
    lengths = rng.integers(0, max_len + 1, size=n_docs)
    w, inp = _packed(lengths, H, 64, 64, seed=31 + n_docs)
    gpu = run_gpu(to_device(inp), w.b, w.mode)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))


def test_many_documents_cut_into_segments():
    rng = np.random.default_rng(7)
    lengths = rng.integers(0, 700, size=50)
    lengths[[3, 17]] = 0
    w, inp = _packed(lengths, 2, 64, 64, seed=41)
    bdla.set_seq_split(1)
    try:
        gpu = run_gpu(to_device(inp), w.b, w.mode)
    finally:
        bdla.set_seq_split(0)
    compare_all(gpu, run_oracle(inp, w.b, w.mode))
