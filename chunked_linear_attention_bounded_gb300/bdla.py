"""Thin ctypes binding of libbdla.so (see include/bdla.h).

Argument marshalling only: shape/dtype checks, output and workspace
allocation through PyTorch (device memory and streams are all PyTorch is used
for), and one C-ABI call per op.  Every arithmetic step runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbdla.so")

BOUNDED = 0    # BDLA_DECAY_BOUNDED_SIGMOID: log g = b * sigmoid(a)
SOFTPLUS = 1   # BDLA_DECAY_NEG_SOFTPLUS:    log g = -softplus(a)   (ablation)
CHUNK = 16
OP_FWD, OP_BWD, OP_DECAY = 0, 1, 2

# bdla_status values (include/bdla.h)
OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_RANGE, ERR_UNSUPPORTED = 0, 1, 2, 3, 4, 5, 6
ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE, ERR_TOO_LARGE = 7, 8, 9, 10, 11
STATUS_NAMES = {OK: "BDLA_OK", ERR_NULL: "BDLA_ERR_NULL", ERR_SHAPE: "BDLA_ERR_SHAPE",
                ERR_DTYPE: "BDLA_ERR_DTYPE", ERR_ALIGN: "BDLA_ERR_ALIGN", ERR_RANGE: "BDLA_ERR_RANGE",
                ERR_UNSUPPORTED: "BDLA_ERR_UNSUPPORTED", ERR_WORKSPACE: "BDLA_ERR_WORKSPACE",
                ERR_CUDA: "BDLA_ERR_CUDA", ERR_TIMEOUT: "BDLA_ERR_TIMEOUT", ERR_DEVICE: "BDLA_ERR_DEVICE",
                ERR_TOO_LARGE: "BDLA_ERR_TOO_LARGE"}

# Every symbol include/*.h declares.
EXPORTS = ("bdla_workspace_bytes", "bdla_decay", "bdla_fwd", "bdla_fwd_varlen", "bdla_bwd",
           "bdla_bwd_varlen", "bdla_read_device_status", "bdla_status_string", "bdla_version",
           "bdla_set_kernel_events", "bdla_fwd_noalloc", "bdla_noalloc_read_status",
           "bdla_set_seq_split", "bdla_decode", "bdla_set_wait_limit_ns", "bdla_set_test_stall",
           "bdla_workspace_bytes_vec", "bdla_fwd_vec", "bdla_bwd_vec", "bdla_workspace_bytes_delta",
           "bdla_fwd_delta", "bdla_bwd_delta", "bdla_tile_states_bytes")
KERNEL_DECAY, KERNEL_FWD, KERNEL_BWD, KERNEL_STATES, KERNEL_SEG = 0, 1, 2, 3, 4
STALL_NONE, STALL_PRODUCER, STALL_MMA, STALL_EPILOGUE = 0, 1, 2, 3


class BdlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int)]


_lib = None


def lib():
    """Loads libbdla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbdla.so is not built ({LIB_PATH}); run "
                               "chunked_linear_attention_bounded_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, f32, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_float, ctypes.c_int
        L.bdla_workspace_bytes.argtypes = [ci, Dims, ci, ci, ci]
        L.bdla_workspace_bytes.restype = sz
        L.bdla_decay.argtypes = [vp, f32, ci, vp, ci, vp, Dims, ci, vp, sz, vp]
        L.bdla_fwd.argtypes = [vp, vp, vp, vp, f32, ci, vp, vp, ci, vp, vp, ci, ci, Dims, ci, vp, sz,
                               vp]
        L.bdla_fwd_varlen.argtypes = [vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, ci, vp, vp, ci, ci, Dims,
                                      ci, vp, sz, vp]
        L.bdla_bwd.argtypes = [vp, vp, vp, vp, f32, ci, vp, vp, vp, vp, ci, ci, vp, vp, vp, vp, vp, Dims,
                               ci, vp, sz, vp]
        L.bdla_bwd_varlen.argtypes = [vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, vp, vp, ci, ci, vp, vp, vp,
                                      vp, vp, Dims, ci, vp, sz, vp]
        for name in ("bdla_decay", "bdla_fwd", "bdla_fwd_varlen", "bdla_bwd", "bdla_bwd_varlen",
                     "bdla_read_device_status", "bdla_noalloc_read_status"):
            getattr(L, name).restype = ci
        L.bdla_read_device_status.argtypes = [vp, vp]
        L.bdla_noalloc_read_status.argtypes = [vp]
        L.bdla_status_string.argtypes = [ci]
        L.bdla_status_string.restype = ctypes.c_char_p
        L.bdla_version.restype = ci
        L.bdla_set_kernel_events.argtypes = [ci, vp, vp]
        L.bdla_set_kernel_events.restype = ci
        L.bdla_fwd_noalloc.argtypes = [vp, vp, vp, vp, f32, ci, vp, vp, ci, vp, Dims, ci, vp]
        L.bdla_fwd_noalloc.restype = ci
        L.bdla_set_seq_split.argtypes = [ci]
        L.bdla_set_seq_split.restype = ci
        L.bdla_decode.argtypes = [vp, vp, vp, vp, f32, vp, vp, ci, Dims, ci, vp]
        L.bdla_decode.restype = ci
        L.bdla_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.bdla_set_wait_limit_ns.restype = ci
        L.bdla_set_test_stall.argtypes = [ci, ci]
        L.bdla_set_test_stall.restype = ci
        L.bdla_workspace_bytes_vec.argtypes = [ci, Dims, ci]
        L.bdla_workspace_bytes_vec.restype = sz
        L.bdla_fwd_vec.argtypes = [vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, ci, vp, vp, Dims, ci, vp, sz, vp]
        L.bdla_fwd_vec.restype = ci
        L.bdla_bwd_vec.argtypes = [vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, Dims,
                                   ci, vp, sz, vp]
        L.bdla_bwd_vec.restype = ci
        L.bdla_workspace_bytes_delta.argtypes = [ci, Dims, ci]
        L.bdla_workspace_bytes_delta.restype = sz
        L.bdla_fwd_delta.argtypes = [vp, vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, ci, vp, vp, Dims, ci, vp, sz,
                                     vp]
        L.bdla_fwd_delta.restype = ci
        L.bdla_bwd_delta.argtypes = [vp, vp, vp, vp, vp, f32, ci, vp, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     Dims, ci, vp, sz, vp]
        L.bdla_tile_states_bytes.argtypes = [Dims, ci]
        L.bdla_tile_states_bytes.restype = sz
        L.bdla_bwd_delta.restype = ci
        del i32
        _lib = L
    return _lib


def set_kernel_events(kernel: int, start=None, stop=None):
    """Measurement hook: record torch.cuda.Event `start`/`stop` around every
    later launch of `kernel` (KERNEL_*); pass None to clear."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    st = lib().bdla_set_kernel_events(int(kernel), h(start), h(stop))
    if st:
        raise BdlaError(st, "bdla_set_kernel_events")


def set_wait_limit_ns(ns: int):
    """Limit of the kernels' pipeline waits for later launches (0 = the
    default 2 s); a test hook (include/bdla_tuning.h)."""
    lib().bdla_set_wait_limit_ns(int(ns))


def set_test_stall(kernel: int, role: int):
    """Test hook: `role` (STALL_*) of `kernel` (KERNEL_*) waits on a barrier
    nothing arrives at, so the bounded wait runs out (STALL_NONE clears)."""
    st = lib().bdla_set_test_stall(int(kernel), int(role))
    if st:
        raise BdlaError(st, "bdla_set_test_stall")


_seq_split = 0


def set_seq_split(blocks: int):
    """Sequence segments of 128-token blocks: 0 automatic, < 0 never, > 0
    always this many blocks per segment (process-wide)."""
    global _seq_split
    lib().bdla_set_seq_split(int(blocks))
    _seq_split = int(blocks)


def segments_engaged(q_shape, dv: int, n_docs: int = 0) -> bool:
    """Whether calls of this shape cut documents into segments under the
    current setting (the segment buffers then appear in the workspace)."""
    cur = _seq_split
    with_cut = workspace_bytes(OP_FWD, q_shape, dv, n_docs)
    set_seq_split(-1)
    try:
        return with_cut > workspace_bytes(OP_FWD, q_shape, dv, n_docs)
    finally:
        set_seq_split(cur)


def status_string(s: int) -> str:
    try:
        return lib().bdla_status_string(int(s)).decode()
    except Exception:  # pragma: no cover
        return "?"


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q: torch.Tensor, v: torch.Tensor) -> Dims:
    B, T, H, dk = q.shape
    return Dims(B, T, H, dk, v.shape[-1])


def n_slots(tokens: int, n_docs: int, stride: int) -> int:
    """Checkpoint slots for `tokens` packed tokens in `n_docs` documents."""
    return (tokens + stride - 1) // stride + n_docs


class Workspace:
    """Caller-owned device scratch for the library (status word first)."""

    def __init__(self, nbytes: int, device):
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def ensure(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device)
        return self

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def read_device_status(self, stream=None) -> int:
        return int(lib().bdla_read_device_status(self.ptr, _stream_handle(stream)))


def workspace_bytes(op: int, q_shape, dv: int, n_docs: int = 0, mode: int = BOUNDED,
                    ckpt_stride: int = 0) -> int:
    B, T, H, dk = q_shape
    return int(lib().bdla_workspace_bytes(op, Dims(B, T, H, dk, dv), n_docs, mode, ckpt_stride))


def _ws_for(op, q, v, n_docs, mode, ckpt_stride, ws: Optional[Workspace]) -> Workspace:
    need = workspace_bytes(op, tuple(q.shape), v.shape[-1], n_docs, mode, ckpt_stride)
    if need == 0:
        raise BdlaError(ERR_SHAPE, "bdla_workspace_bytes")
    if ws is None:
        return Workspace(need, q.device)
    return ws.ensure(need)


def decay(a: torch.Tensor, b: float = -5.0, cu_seqlens: Optional[torch.Tensor] = None,
          mode: int = BOUNDED, ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """Tile-local inclusive cumsum Gamma of the log-decay, fp32 [H, B*T]
    (head-major)."""
    _check(a, "a", torch.float32, 3)
    B, T, H = a.shape
    gamma = torch.empty((H, B * T), dtype=torch.float32, device=a.device)
    n_docs = 0
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
        n_docs = cu_seqlens.numel() - 1
    ws = ws or Workspace(256, a.device)
    st = lib().bdla_decay(_p(a), b, CHUNK, _p(cu_seqlens), n_docs, _p(gamma),
                          Dims(B, T, H, 64, 64), mode, ws.ptr, ws.nbytes, _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_decay")
    return gamma


def decode(q, k, v, a, state, b: float = -5.0, mode: int = BOUNDED, o_dtype=torch.bfloat16,
           out=None, stream=None) -> torch.Tensor:
    """One recurrent step per sequence: q, k [B, H, dk], v [B, H, dv] bf16,
    a [B, H] fp32; `state` fp32 [B, H, dk, dv] is updated in place
    (S <- e^{lambda} S + k v^T).  Returns o = S^T q [B, H, dv]."""
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3)
    _check(a, "a", torch.float32, 2)
    _check(state, "state", torch.float32, 4)
    B, H, dk = q.shape
    dv = v.shape[-1]
    if tuple(state.shape) != (B, H, dk, dv) or tuple(a.shape) != (B, H):
        raise BdlaError(ERR_SHAPE, "decode shapes")
    o = out if out is not None else torch.empty((B, H, dv), dtype=o_dtype, device=q.device)
    st = lib().bdla_decode(_p(q), _p(k), _p(v), _p(a), b, _p(state), _p(o), _dtype_code(o.dtype),
                           Dims(B, 1, H, dk, dv), mode, _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_decode")
    return o


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return 0
    if dt == torch.float32:
        return 1
    raise ValueError(f"unsupported dtype {dt}")


def fwd(q, k, v, a, b: float = -5.0, h0=None, cu_seqlens=None, mode: int = BOUNDED,
        o_dtype=torch.bfloat16, want_hT: bool = True, ckpt_stride: int = 0,
        ckpt_dtype=torch.float32, ws: Optional[Workspace] = None, out=None, hT_out=None,
        ckpt_out=None, stream=None):
    """Forward pass.  Returns (o, hT, ckpt); hT / ckpt are None when not asked
    for.  ckpt_stride > 0 also writes the state every ckpt_stride tokens
    ([H, n_slots, dk, dv], ckpt_dtype), which bwd() can reuse."""
    _check(q, "q", torch.bfloat16, 4)
    _check(k, "k", torch.bfloat16, 4)
    _check(v, "v", torch.bfloat16, 4)
    _check(a, "a", torch.float32, 3)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or a.shape != q.shape[:3]:
        raise ValueError("q, k, v, a shapes disagree")
    n_docs = 0
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
        n_docs = cu_seqlens.numel() - 1
    n_seq = n_docs if n_docs else B
    if h0 is not None:
        _check(h0, "h0", torch.float32, 4)
        if tuple(h0.shape) != (n_seq, H, dk, dv):
            raise ValueError("h0 must be [n_docs, H, dk, dv]")
    dev = q.device
    o = out if out is not None else torch.empty((B, T, H, dv), dtype=o_dtype, device=dev)
    hT = hT_out
    if hT is None and want_hT:
        hT = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev)
    ckpt = ckpt_out
    if ckpt is None and ckpt_stride:
        ckpt = torch.empty((H, n_slots(B * T, n_seq, ckpt_stride), dk, dv), dtype=ckpt_dtype,
                           device=dev)
    ws = _ws_for(OP_FWD, q, v, n_docs, mode, 0, ws)
    odt = 1 if o.dtype == torch.float32 else 0
    ckdt = _dtype_code(ckpt.dtype) if ckpt is not None else 1
    args_tail = (_p(h0), _p(o), odt, _p(hT), _p(ckpt), int(ckpt_stride), ckdt, _dims(q, v), mode,
                 ws.ptr, ws.nbytes, _stream_handle(stream))
    L = lib()
    if n_docs:
        st = L.bdla_fwd_varlen(_p(q), _p(k), _p(v), _p(a), b, CHUNK, _p(cu_seqlens), n_docs,
                               *args_tail)
    else:
        st = L.bdla_fwd(_p(q), _p(k), _p(v), _p(a), b, CHUNK, *args_tail)
    if st:
        raise BdlaError(st, "bdla_fwd")
    return o, hT, ckpt


def bwd(q, k, v, a, dO, b: float = -5.0, h0=None, dhT=None, cu_seqlens=None, ckpt=None,
        ckpt_stride: int = 0, mode: int = BOUNDED, want_dh0: bool = False,
        ws: Optional[Workspace] = None, outs=None, stream=None):
    """Backward pass.  Returns (dq, dk, dv, da, dh0); dh0 is None unless asked for."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dO, "dO")):
        _check(t, n, torch.bfloat16, 4)
    _check(a, "a", torch.float32, 3)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if dO.shape != v.shape:
        raise ValueError("dO must match v")
    n_docs = 0
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
        n_docs = cu_seqlens.numel() - 1
    n_seq = n_docs if n_docs else B
    for t, n in ((h0, "h0"), (dhT, "dhT")):
        if t is not None:
            _check(t, n, torch.float32, 4)
            if tuple(t.shape) != (n_seq, H, dk, dv):
                raise ValueError(f"{n} must be [n_docs, H, dk, dv]")
    ckdt = 1
    if ckpt is not None:
        _check(ckpt, "ckpt", ckpt.dtype, 4)
        ckdt = _dtype_code(ckpt.dtype)
        if not ckpt_stride:
            raise ValueError("ckpt needs its ckpt_stride")
    dev = q.device
    if outs is None:
        dq = torch.empty((B, T, H, dk), dtype=torch.float32, device=dev)
        dkk = torch.empty((B, T, H, dk), dtype=torch.float32, device=dev)
        dvv = torch.empty((B, T, H, dv), dtype=torch.float32, device=dev)
        da = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    else:
        dq, dkk, dvv, da = outs
    dh0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev) if want_dh0 else None
    stride = int(ckpt_stride) if ckpt is not None else 0
    ws_stride = stride if (ckdt == 1 or dv <= 128) else 0
    ws = _ws_for(OP_BWD, q, v, n_docs, mode, ws_stride, ws)
    args_tail = (_p(h0), _p(dO), _p(dhT), _p(ckpt), stride, ckdt, _p(dq), _p(dkk), _p(dvv), _p(da),
                 _p(dh0), _dims(q, v), mode, ws.ptr, ws.nbytes, _stream_handle(stream))
    L = lib()
    if n_docs:
        st = L.bdla_bwd_varlen(_p(q), _p(k), _p(v), _p(a), b, CHUNK, _p(cu_seqlens), n_docs,
                               *args_tail)
    else:
        st = L.bdla_bwd(_p(q), _p(k), _p(v), _p(a), b, CHUNK, *args_tail)
    if st:
        raise BdlaError(st, "bdla_bwd")
    return dq, dkk, dvv, da, dh0


# ---------------------------------------------------------------- per-channel decay
def _vec_checks(q, k, v, a, cu_seqlens, h0):
    _check(q, "q", torch.bfloat16, 4)
    _check(k, "k", torch.bfloat16, 4)
    _check(v, "v", torch.bfloat16, 4)
    _check(a, "a", torch.float32, 4)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or a.shape != q.shape:
        raise ValueError("q, k, v, a shapes disagree (a is [B, T, H, dk] for per-channel decay)")
    n_docs = 0
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
        n_docs = cu_seqlens.numel() - 1
    n_seq = n_docs if n_docs else B
    if h0 is not None:
        _check(h0, "h0", torch.float32, 4)
        if tuple(h0.shape) != (n_seq, H, dk, dv):
            raise ValueError("h0 must be [n_docs, H, dk, dv]")
    return B, T, H, dk, dv, n_docs, n_seq


def _ws_vec(op, q, v, n_docs, ws):
    B, T, H, dk = q.shape
    need = int(lib().bdla_workspace_bytes_vec(op, Dims(B, T, H, dk, v.shape[-1]), n_docs))
    if need == 0:
        raise BdlaError(ERR_UNSUPPORTED, "bdla_workspace_bytes_vec")
    if ws is None:
        return Workspace(need, q.device)
    return ws.ensure(need)


def tile_states(q, v, cu_seqlens=None):
    """An uninitialised bf16 buffer for the state before every 16-token tile
    ([H, slots, dk, dv]), the `states` hand-off of the per-channel and
    delta-rule paths."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n_docs = cu_seqlens.numel() - 1 if cu_seqlens is not None else 0
    nbytes = int(lib().bdla_tile_states_bytes(Dims(B, T, H, dk, dv), n_docs))
    if nbytes == 0:
        raise BdlaError(ERR_UNSUPPORTED, "bdla_tile_states_bytes")
    return torch.empty((H, nbytes // (2 * H * dk * dv), dk, dv), dtype=torch.bfloat16, device=q.device)


def fwd_vec(q, k, v, a, b: float = -5.0, h0=None, cu_seqlens=None, mode: int = BOUNDED,
            o_dtype=torch.bfloat16, ws: Optional[Workspace] = None, states_out=None, stream=None):
    """Forward pass with one log-decay per key channel (a [B, T, H, dk]).
    Returns (o, hT); with `states_out` (from tile_states) it also writes the
    state before every tile there, for bwd_vec."""
    B, T, H, dk, dv, n_docs, n_seq = _vec_checks(q, k, v, a, cu_seqlens, h0)
    o = torch.empty((B, T, H, dv), dtype=o_dtype, device=q.device)
    hT = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _ws_vec(OP_FWD, q, v, n_docs, ws)
    st = lib().bdla_fwd_vec(_p(q), _p(k), _p(v), _p(a), b, CHUNK, _p(cu_seqlens), n_docs, _p(h0), _p(o),
                            _dtype_code(o.dtype), _p(hT), _p(states_out), _dims(q, v), mode, ws.ptr, ws.nbytes,
                            _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_fwd_vec")
    return o, hT


def bwd_vec(q, k, v, a, dO, b: float = -5.0, h0=None, dhT=None, cu_seqlens=None, mode: int = BOUNDED,
            want_dh0: bool = False, ws: Optional[Workspace] = None, outs=None, states=None, stream=None):
    """Backward pass with one log-decay per key channel.  Returns
    (dq, dk, dv, da, dh0) with da [B, T, H, dk]; dh0 is None unless asked for."""
    B, T, H, dk, dv, n_docs, n_seq = _vec_checks(q, k, v, a, cu_seqlens, h0)
    _check(dO, "dO", torch.bfloat16, 4)
    if dO.shape != v.shape:
        raise ValueError("dO must match v")
    if dhT is not None:
        _check(dhT, "dhT", torch.float32, 4)
    dev = q.device
    if outs is None:
        outs = (torch.empty(q.shape, dtype=torch.float32, device=dev),
                torch.empty(k.shape, dtype=torch.float32, device=dev),
                torch.empty(v.shape, dtype=torch.float32, device=dev),
                torch.empty(a.shape, dtype=torch.float32, device=dev))
    dq, dk_, dv_, da = outs
    dh0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev) if want_dh0 else None
    ws = _ws_vec(OP_BWD, q, v, n_docs, ws)
    st = lib().bdla_bwd_vec(_p(q), _p(k), _p(v), _p(a), b, CHUNK, _p(cu_seqlens), n_docs, _p(h0), _p(dO),
                            _p(dhT), _p(states), _p(dq), _p(dk_), _p(dv_), _p(da), _p(dh0), _dims(q, v), mode,
                            ws.ptr, ws.nbytes, _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_bwd_vec")
    return dq, dk_, dv_, da, dh0


# ---------------------------------------------------------------- gated delta rule
def _delta_checks(q, k, v, a, beta, cu_seqlens, h0):
    _check(q, "q", torch.bfloat16, 4)
    _check(k, "k", torch.bfloat16, 4)
    _check(v, "v", torch.bfloat16, 4)
    _check(a, "a", torch.float32, 3)
    _check(beta, "beta", torch.float32, 3)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or a.shape != q.shape[:3] or beta.shape != a.shape:
        raise ValueError("q, k, v, a, beta shapes disagree")
    n_docs = 0
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, 1)
        n_docs = cu_seqlens.numel() - 1
    n_seq = n_docs if n_docs else B
    if h0 is not None:
        _check(h0, "h0", torch.float32, 4)
        if tuple(h0.shape) != (n_seq, H, dk, dv):
            raise ValueError("h0 must be [n_docs, H, dk, dv]")
    return B, T, H, dk, dv, n_docs, n_seq


def _ws_delta(op, q, v, n_docs, ws):
    B, T, H, dk = q.shape
    need = int(lib().bdla_workspace_bytes_delta(op, Dims(B, T, H, dk, v.shape[-1]), n_docs))
    if need == 0:
        raise BdlaError(ERR_UNSUPPORTED, "bdla_workspace_bytes_delta")
    if ws is None:
        return Workspace(need, q.device)
    return ws.ensure(need)


def fwd_delta(q, k, v, a, beta, b: float = -5.0, h0=None, cu_seqlens=None, mode: int = BOUNDED,
              o_dtype=torch.bfloat16, ws: Optional[Workspace] = None, out=None, hT_out=None, states_out=None,
              stream=None):
    """Gated delta rule forward (a, beta [B, T, H]).  Returns (o, hT); with
    `states_out` (from tile_states) it also writes the state before every
    tile there, for bwd_delta."""
    B, T, H, dk, dv, n_docs, n_seq = _delta_checks(q, k, v, a, beta, cu_seqlens, h0)
    o = out if out is not None else torch.empty((B, T, H, dv), dtype=o_dtype, device=q.device)
    hT = hT_out if hT_out is not None else torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = _ws_delta(OP_FWD, q, v, n_docs, ws)
    st = lib().bdla_fwd_delta(_p(q), _p(k), _p(v), _p(a), _p(beta), b, CHUNK, _p(cu_seqlens), n_docs, _p(h0),
                              _p(o), _dtype_code(o.dtype), _p(hT), _p(states_out), _dims(q, v), mode, ws.ptr,
                              ws.nbytes, _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_fwd_delta")
    return o, hT


def bwd_delta(q, k, v, a, beta, dO, b: float = -5.0, h0=None, dhT=None, cu_seqlens=None, mode: int = BOUNDED,
              want_dh0: bool = False, ws: Optional[Workspace] = None, outs=None, states=None, stream=None):
    """Gated delta rule backward.  Returns (dq, dk, dv, da, dbeta, dh0);
    dh0 is None unless asked for."""
    B, T, H, dk, dv, n_docs, n_seq = _delta_checks(q, k, v, a, beta, cu_seqlens, h0)
    _check(dO, "dO", torch.bfloat16, 4)
    if dO.shape != v.shape:
        raise ValueError("dO must match v")
    if dhT is not None:
        _check(dhT, "dhT", torch.float32, 4)
    dev = q.device
    if outs is None:
        outs = (torch.empty(q.shape, dtype=torch.float32, device=dev),
                torch.empty(k.shape, dtype=torch.float32, device=dev),
                torch.empty(v.shape, dtype=torch.float32, device=dev),
                torch.empty(a.shape, dtype=torch.float32, device=dev),
                torch.empty(beta.shape, dtype=torch.float32, device=dev))
    dq, dk_, dv_, da, dbeta = outs
    dh0 = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device=dev) if want_dh0 else None
    ws = _ws_delta(OP_BWD, q, v, n_docs, ws)
    st = lib().bdla_bwd_delta(_p(q), _p(k), _p(v), _p(a), _p(beta), b, CHUNK, _p(cu_seqlens), n_docs, _p(h0),
                              _p(dO), _p(dhT), _p(states), _p(dq), _p(dk_), _p(dv_), _p(da), _p(dbeta), _p(dh0),
                              _dims(q, v), mode, ws.ptr, ws.nbytes, _stream_handle(stream))
    if st:
        raise BdlaError(st, "bdla_bwd_delta")
    return dq, dk_, dv_, da, dbeta, dh0
