"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/bdla.h declares, sizes its workspace, and rejects bad arguments on
the host before any launch."""
import ctypes
import os
import re

import pytest

import chunked_linear_attention_bounded_gb300 as pkg
from chunked_linear_attention_bounded_gb300 import bdla
from chunked_linear_attention_bounded_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return bdla.lib()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(bdla_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert declared == set(bdla.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    for code in range(12):
        assert bdla.status_string(code) not in ("", "unknown status")
    assert bdla.status_string(123) == "unknown status"
    assert L.bdla_version() >= 100


def test_workspace_bytes(L):
    fwd = bdla.workspace_bytes(bdla.OP_FWD, (1, 65536, 32, 128), 128, n_docs=8)
    assert fwd >= 256 + 65536 * 32 * 4
    bwd = bdla.workspace_bytes(bdla.OP_BWD, (1, 65536, 32, 128), 128, n_docs=8)
    bwd16 = bdla.workspace_bytes(bdla.OP_BWD, (1, 65536, 32, 128), 128, n_docs=8, ckpt_stride=16)
    bwd128 = bdla.workspace_bytes(bdla.OP_BWD, (1, 65536, 32, 128), 128, n_docs=8, ckpt_stride=128)
    # without checkpoints the backward recomputes bf16 block states; with fp32
    # checkpoints inside the blocks it converts their block starts into the same
    # array; block checkpoints are read as they are
    states = 32 * (65536 // 128 + 8) * 128 * 128 * 2
    assert bwd == bwd16 == bwd128 + states
    assert bwd128 >= fwd
    assert bdla.workspace_bytes(bdla.OP_FWD, (1, 16, 2, 96), 64) == 0      # dk 96 unsupported
    assert bdla.workspace_bytes(bdla.OP_FWD, (1, 16, 2, 64), 32) == 0      # dv 32 unsupported


# Non-NULL, aligned, never dereferenced: every call below is rejected by a host
# check before any launch (none of them may reach a kernel).
FAKE = ctypes.c_void_p(1 << 20)


def _fwd(L, b=-5.0, chunk=16, dims=(1, 64, 2, 64, 64), mode=0, q=FAKE, ws=FAKE, ws_bytes=1 << 40,
         ckpt=None, stride=0, o_dtype=0, ck_dtype=1):
    return L.bdla_fwd(q, FAKE, FAKE, FAKE, b, chunk, None, FAKE, o_dtype, None, ckpt, stride, ck_dtype,
                      bdla.Dims(*dims), mode, ws, ws_bytes, None)


def test_segment_buffers_size_the_workspace(L):
    """Cutting documents into segments adds the per-segment state buffer
    (slots x H x dk x dv fp32) to the workspace in place of the small
    document-order array; the plan uses sizes only."""
    shape = (1, 8192, 4, 128)
    try:
        bdla.set_seq_split(-1)
        plain = bdla.workspace_bytes(bdla.OP_BWD, shape, 128, n_docs=2)
        bdla.set_seq_split(4)                 # 512-token segments
        cut = bdla.workspace_bytes(bdla.OP_BWD, shape, 128, n_docs=2)
        slots = 8192 // 512 + 2
        assert cut - plain >= slots * 4 * 128 * 128 * 4
        bdla.set_seq_split(0)                 # 2 x 4 units: fewer than the SMs, cut
        assert bdla.workspace_bytes(bdla.OP_BWD, shape, 128, n_docs=2) > plain
        many = (1, 8192, 128, 128)            # 2 x 128 units: no cut
        bdla.set_seq_split(-1)
        m_plain = bdla.workspace_bytes(bdla.OP_BWD, many, 128, n_docs=2)
        bdla.set_seq_split(0)
        assert bdla.workspace_bytes(bdla.OP_BWD, many, 128, n_docs=2) == m_plain
    finally:
        bdla.set_seq_split(0)


def test_decode_host_validation(L):
    """bdla_decode refuses bad arguments before any launch (fake pointers are
    never dereferenced)."""
    fake = ctypes.c_void_p(1 << 20)
    call = lambda dims, b=-5.0, mode=0, ptr=fake, odt=0: L.bdla_decode(
        ptr, fake, fake, fake, b, fake, fake, odt, dims, mode, None)
    assert call(bdla.Dims(4, 2, 2, 128, 128)) == bdla.ERR_SHAPE          # T must be 1
    assert call(bdla.Dims(4, 1, 2, 96, 128)) == bdla.ERR_UNSUPPORTED     # dk 96 unsupported
    assert call(bdla.Dims(4, 1, 2, 128, 128), b=0.5) == bdla.ERR_RANGE   # b > 0
    assert call(bdla.Dims(4, 1, 2, 128, 128), ptr=None) == bdla.ERR_NULL
    assert call(bdla.Dims(4, 1, 2, 128, 128), ptr=ctypes.c_void_p((1 << 20) + 4)) == bdla.ERR_ALIGN
    assert call(bdla.Dims(4, 1, 2, 128, 128), odt=7) == bdla.ERR_DTYPE


def test_host_validation_before_launch(L):
    E = bdla
    assert _fwd(L, chunk=32) == E.ERR_UNSUPPORTED              # chunk != 16
    assert _fwd(L, b=0.5) == E.ERR_RANGE                       # b > 0
    assert _fwd(L, b=float("nan")) == E.ERR_RANGE
    assert _fwd(L, b=-5.5) == E.ERR_RANGE                      # 16 * 5.5 > 80
    assert _fwd(L, b=-9.0, mode=1, ws_bytes=16) == E.ERR_WORKSPACE   # ablation ignores b
    assert _fwd(L, mode=7) == E.ERR_UNSUPPORTED
    assert _fwd(L, dims=(1, 64, 2, 96, 64)) == E.ERR_UNSUPPORTED
    assert _fwd(L, dims=(1, 64, 2, 256, 64)) == E.ERR_UNSUPPORTED   # dk = 256 refused
    assert _fwd(L, dims=(1, -1, 2, 64, 64)) == E.ERR_SHAPE
    assert _fwd(L, dims=(0, 64, 2, 64, 64)) == E.ERR_SHAPE
    assert _fwd(L, dims=(65536, 1, 1, 64, 64)) == E.ERR_UNSUPPORTED  # documents are a grid extent
    assert _fwd(L, q=None) == E.ERR_NULL
    assert _fwd(L, q=ctypes.c_void_p((1 << 20) + 8)) == E.ERR_ALIGN
    assert _fwd(L, ws=None) == E.ERR_WORKSPACE
    assert _fwd(L, ws_bytes=16) == E.ERR_WORKSPACE
    assert _fwd(L, ckpt=FAKE, stride=24) == E.ERR_SHAPE
    assert _fwd(L, o_dtype=5) == E.ERR_DTYPE
    assert _fwd(L, ckpt=FAKE, stride=64, ck_dtype=0) == E.ERR_UNSUPPORTED   # bf16 needs stride % 128 == 0
    assert _fwd(L, ckpt=FAKE, stride=128, ck_dtype=7) == E.ERR_DTYPE
    st = L.bdla_bwd(FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, None, None, None, 0, 1, FAKE, FAKE, FAKE,
                    FAKE, None, bdla.Dims(1, 64, 2, 64, 64), 0, FAKE, 1 << 40, None)
    assert st == E.ERR_NULL                                    # dO missing
    st = L.bdla_bwd(FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, FAKE, None, FAKE, 128, 9, FAKE, FAKE, FAKE,
                    FAKE, None, bdla.Dims(1, 64, 2, 64, 64), 0, FAKE, 1 << 40, None)
    assert st == E.ERR_DTYPE                                   # checkpoint dtype 9
    st = L.bdla_fwd_varlen(FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, 2, None, FAKE, 0, None, None, 0, 1,
                           bdla.Dims(1, 64, 2, 64, 64), 0, FAKE, 1 << 40, None)
    assert st == E.ERR_NULL                                    # cu_seqlens missing
    st = L.bdla_fwd_varlen(FAKE, FAKE, FAKE, FAKE, -5.0, 16, FAKE, 2, None, FAKE, 0, None, None, 0, 1,
                           bdla.Dims(2, 64, 2, 64, 64), 0, FAKE, 1 << 40, None)
    assert st == E.ERR_SHAPE                                   # varlen needs B == 1


def test_segment_plan_with_the_largest_document_count(L):
    """65535 documents (the grid limit) leave no room for segment slots: a
    forced cut is then skipped instead of dividing by zero while planning."""
    try:
        bdla.set_seq_split(1)
        n = bdla.workspace_bytes(bdla.OP_FWD, (1, 65535 * 2, 1, 64), 64, n_docs=65535)
        bdla.set_seq_split(-1)
        assert n == bdla.workspace_bytes(bdla.OP_FWD, (1, 65535 * 2, 1, 64), 64, n_docs=65535) > 0
    finally:
        bdla.set_seq_split(0)


def test_package_exports():
    for name in ("fwd", "bwd", "decay", "Workspace", "BdlaError"):
        assert hasattr(pkg, name)


def test_variant_workspace_and_tile_states_sizes(L):
    """Per-channel / delta-rule calls: the state before every 16-token tile
    takes H x (tokens/16 + documents + 1) bf16 dk x dv matrices; packed calls
    with several documents also keep the documents' launch order (one int32
    each) in the workspace; the backward's workspace adds its own states."""
    D = bdla.Dims(1, 65536, 32, 128, 128)
    slots = 65536 // 16 + 8 + 1
    assert L.bdla_tile_states_bytes(D, 8) == 32 * slots * 128 * 128 * 2
    assert L.bdla_tile_states_bytes(bdla.Dims(2, 100, 3, 64, 64), 0) == 3 * (200 // 16 + 2 + 1) * 64 * 64 * 2
    assert L.bdla_tile_states_bytes(bdla.Dims(1, 16, 2, 128, 256), 0) == 0       # dv 256 unsupported here
    for ws_fn in (L.bdla_workspace_bytes_vec, L.bdla_workspace_bytes_delta):
        f_packed = ws_fn(bdla.OP_FWD, D, 8)
        f_one = ws_fn(bdla.OP_FWD, D, 1)
        f_fixed = ws_fn(bdla.OP_FWD, bdla.Dims(8, 8192, 32, 128, 128), 0)
        assert f_packed > f_one == f_fixed                 # the order region (8 documents)
        b_packed = ws_fn(bdla.OP_BWD, D, 8)
        assert b_packed - f_packed >= L.bdla_tile_states_bytes(D, 8)


def test_variant_host_validation(L):
    """The per-channel and delta-rule entry points refuse bad arguments on the
    host (nothing below reaches a kernel)."""
    E = bdla
    Dm = bdla.Dims(1, 64, 2, 64, 64)
    st = L.bdla_fwd_vec(FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, 0, None, FAKE, 0, None,
                        ctypes.c_void_p((1 << 20) + 8), Dm, 0, FAKE, 1 << 40, None)
    assert st == E.ERR_ALIGN                                   # misaligned states
    st = L.bdla_fwd_delta(FAKE, FAKE, FAKE, FAKE, None, -5.0, 16, None, 0, None, FAKE, 0, None, None, Dm, 0,
                          FAKE, 1 << 40, None)
    assert st == E.ERR_NULL                                    # beta missing
    st = L.bdla_bwd_delta(FAKE, FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, 0, None, FAKE, None, None, FAKE, FAKE,
                          FAKE, FAKE, None, None, Dm, 0, FAKE, 1 << 40, None)
    assert st == E.ERR_NULL                                    # dbeta missing
    st = L.bdla_fwd_delta(FAKE, FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, 0, None, FAKE, 0, None, None,
                          bdla.Dims(1, 64, 2, 64, 256), 0, FAKE, 1 << 40, None)
    assert st == E.ERR_UNSUPPORTED                             # dv 256
    st = L.bdla_fwd_vec(FAKE, FAKE, FAKE, FAKE, -5.0, 16, None, 0, None, FAKE, 0, None, None, Dm, 0, FAKE, 16,
                        None)
    assert st == E.ERR_WORKSPACE
