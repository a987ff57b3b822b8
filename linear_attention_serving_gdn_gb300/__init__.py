"""Gated DeltaNet linear-attention hot path for one GB300 (sm_103a).

A thin ctypes binding over ``libgdn.so`` (C ABI in ``include/gdn.h``).  The
functions below carry the C names; they only check and marshal PyTorch
tensors (dtype, device, contiguity, shapes) into pointers and the current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind: if the library is missing, every entry
point raises.

Layouts (all row-major, device memory):
  q, k        [T][h_k][d_k]  bfloat16
  v, o        [T][h_v][d_v]  bfloat16
  g, beta     [T][h_v]       float32   (alpha = exp(g))
  state       [num_slots][h_v][d_v][d_k] float32   (S^T per slot and head)
  chunk_states [n_emit][h_v][d_v][d_k] float32
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "GdnError", "load_library", "library_path", "prepare_decode_packed",
    "gdn_decode_packed", "gdn_decode_packed_raw", "gdn_prep_inputs", "gdn_decode_multi",
    "gdn_prefill_varlen", "gdn_prefill_varlen_apc", "gdn_mixed_step", "gdn_mixed_step_colaunch", "gdn_prefill_num_emits", "gdn_prefill_emit_offsets", "gdn_align_block_size",
    "gdn_floor_prefix_hit", "gdn_grid_emit_every_chunks", "gdn_status_string",
    "gdn_prefill_workspace_bytes", "gdn_status_from_device",
    "EXPORTED_SYMBOLS", "GDN_DEV_BAD_SLOT", "GDN_DEV_TIMEOUT",
]

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA = 0, 1, 2, 3
GDN_ERR_WORKSPACE, GDN_ERR_TIMEOUT = 4, 5
GDN_DEV_BAD_SLOT, GDN_DEV_TIMEOUT = 0x1, 0x2

EXPORTED_SYMBOLS = (
    "gdn_decode_packed", "gdn_decode_packed_raw", "gdn_prep_inputs", "gdn_decode_multi",
    "gdn_prefill_varlen", "gdn_prefill_varlen_apc", "gdn_mixed_step", "gdn_mixed_step_colaunch", "gdn_prefill_num_emits", "gdn_prefill_emit_offsets", "gdn_align_block_size",
    "gdn_floor_prefix_hit", "gdn_grid_emit_every_chunks", "gdn_status_string",
    "gdn_prefill_workspace_bytes", "gdn_status_from_device",
)


class GdnError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {gdn_status_string(status)}")


class Dims(ctypes.Structure):
    _fields_ = [("h_k", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("scale", ctypes.c_float)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_lib = None


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Load libgdn.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libgdn.so is not built ({_build.LIB}); run __graft_entry__.build()")
    _lib = _configure(ctypes.CDLL(_build.LIB))
    return _lib


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures of every entry point on a loaded library."""
    lib.gdn_decode_packed.restype = ctypes.c_int
    lib.gdn_decode_packed.argtypes = [ctypes.POINTER(Dims), _I32, _P, _P, _P, _P, _P, _P, _I64,
                                      _P, _P, _P, _P, _P]
    lib.gdn_decode_packed_raw.restype = ctypes.c_int
    lib.gdn_decode_packed_raw.argtypes = [ctypes.POINTER(Dims), _I32, _P, _P, _P, _P, _P, _P, _P,
                                          ctypes.c_float, _P, _I64, _P, _P, _P, _P, _P]
    lib.gdn_prep_inputs.restype = ctypes.c_int
    lib.gdn_prep_inputs.argtypes = [ctypes.POINTER(Dims), _I64, _P, _P, _P, _P, _P, _P, ctypes.c_float,
                                    _P, _P, _P, _P, _P]
    lib.gdn_decode_multi.restype = ctypes.c_int
    lib.gdn_decode_multi.argtypes = [ctypes.POINTER(Dims), _I32, _I32, _P, _P, _P, _P, _P, _P, _I64,
                                     _P, _P, _P, _P, _P]
    lib.gdn_prefill_varlen.restype = ctypes.c_int
    lib.gdn_prefill_varlen.argtypes = [ctypes.POINTER(Dims), _I32, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _I64, _P, _P, _P, _P, _I32, _I64, _P, _SZ, _P, _P]
    lib.gdn_prefill_varlen_apc.restype = ctypes.c_int
    lib.gdn_prefill_varlen_apc.argtypes = [ctypes.POINTER(Dims), _I32, _P, _P, _P, _P, _P, _P, _P,
                                           _P, _I64, _P, _P, _P, _I32, _P, _I32, _P, _P, _SZ, _P, _P]
    lib.gdn_mixed_step.restype = ctypes.c_int
    lib.gdn_mixed_step.argtypes = [ctypes.POINTER(Dims), _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _I64, _P, _P, _P, _P, _P, _P, _I32, _I64, _P, _SZ, _P, _P]
    lib.gdn_mixed_step_colaunch.restype = ctypes.c_int
    lib.gdn_mixed_step_colaunch.argtypes = lib.gdn_mixed_step.argtypes + [_P, _P, _P]
    lib.gdn_prefill_workspace_bytes.restype = _SZ
    lib.gdn_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Dims), _I32, _I64]
    lib.gdn_status_from_device.restype = ctypes.c_int
    lib.gdn_status_from_device.argtypes = [_I32]
    lib.gdn_prefill_num_emits.restype = _I64
    lib.gdn_prefill_num_emits.argtypes = [_P, _I32, _I32]
    lib.gdn_prefill_emit_offsets.restype = ctypes.c_int
    lib.gdn_prefill_emit_offsets.argtypes = [_P, _I32, _I32, _P]
    lib.gdn_align_block_size.restype = _I32
    lib.gdn_align_block_size.argtypes = [_I32]
    lib.gdn_floor_prefix_hit.restype = _I64
    lib.gdn_floor_prefix_hit.argtypes = [_I64, _I64, _I32]
    lib.gdn_grid_emit_every_chunks.restype = _I32
    lib.gdn_grid_emit_every_chunks.argtypes = [_I32]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _dev(t, name, dtype, ndim=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    # the common case in one expression; the checks below name what is wrong
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype is dtype and t.is_contiguous()
            and (ndim is None or t.dim() == ndim)):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _ptr(t):
    # a plain int: the argtypes (c_void_p) convert it
    return None if t is None else t.data_ptr()


# The current stream's handle without building a Stream object (a third of
# a small call's Python time); the public route where torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _host_i32(x, name):
    if isinstance(x, torch.Tensor):
        if x.is_cuda:
            raise ValueError(f"{name} must live in host memory")
        x = x.to(torch.int32).contiguous()
        return x, ctypes.c_void_p(x.data_ptr())
    arr = (ctypes.c_int32 * len(x))(*[int(v) for v in x])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def _workspace(ws, dims, num_seqs, total_tokens):
    """(pointer, bytes) of a caller workspace; checks it against the library's need."""
    need = load_library().gdn_prefill_workspace_bytes(ctypes.byref(dims), int(num_seqs), int(total_tokens))
    if ws is None:
        if need:
            raise ValueError(f"this prefill needs a {need}-byte workspace (gdn_prefill_workspace_bytes)")
        return None, 0
    ws = _dev(ws, "workspace", torch.uint8)
    return _ptr(ws), ws.numel()


def _check(status, fn):
    if status != GDN_OK:
        raise GdnError(status, fn)


_dims_cache = {}


def _dims(q, v, scale):
    key = (q.shape[1], v.shape[1], q.shape[2], v.shape[2], float(scale))
    d = _dims_cache.get(key)
    if d is None:  # read-only on the C side, so one object per shape serves every call
        d = _dims_cache[key] = Dims(*key)
    return d


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def gdn_decode_packed(q, k, v, g, beta, state, src_slot, o, dst_slot=None, dev_status=None,
                      scale: float = 1.0, stream=None) -> None:
    """Packed recurrent decode of ``q.shape[0]`` cached rows (see gdn.h)."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    state = _dev(state, "state", f32, 4)
    src_slot = _dev(src_slot, "src_slot", i32, 1)
    dst_slot = _dev(dst_slot, "dst_slot", i32, 1, optional=True)
    o = _dev(o, "o", bf, 3)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    rows = q.shape[0]
    if not (k.shape == q.shape and v.shape[0] == rows and o.shape == v.shape
            and g.shape == (rows, v.shape[1]) and beta.shape == g.shape
            and src_slot.shape[0] == rows and (dst_slot is None or dst_slot.shape[0] == rows)
            and state.shape[1:] == (v.shape[1], v.shape[2], q.shape[2])):
        raise ValueError("inconsistent decode shapes")
    d = _dims(q, v, scale)
    _check(lib.gdn_decode_packed(ctypes.byref(d), rows, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(state), state.shape[0], _ptr(src_slot),
                                 _ptr(dst_slot), _ptr(o), _ptr(dev_status), _stream(stream)),
           "gdn_decode_packed")


class _PreparedCall:
    """A C-ABI call whose arguments were checked and marshalled once: calling
    it issues the same call again on the same buffers (whatever they hold by
    then) and the same stream, with no per-call checks in Python.  The
    buffers must stay alive and keep their shapes and storage."""

    def __init__(self, fn, args, name, keep):
        self._fn, self._args, self._name, self._keep = fn, args, name, keep

    def __call__(self) -> None:
        status = self._fn(*self._args)
        if status != GDN_OK:
            raise GdnError(status, self._name)


def prepare_decode_packed(q, k, v, g, beta, state, src_slot, o, dst_slot=None, dev_status=None,
                          scale: float = 1.0, stream=None) -> _PreparedCall:
    """``gdn_decode_packed`` on fixed buffers, checked once: returns a callable
    that repeats the call (a serving loop refills q, k, v, g, beta and the
    slot lists in place between steps).  The stream is the one given, or the
    current stream at preparation."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    state = _dev(state, "state", f32, 4)
    src_slot = _dev(src_slot, "src_slot", i32, 1)
    dst_slot = _dev(dst_slot, "dst_slot", i32, 1, optional=True)
    o = _dev(o, "o", bf, 3)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    rows = q.shape[0]
    if not (k.shape == q.shape and v.shape[0] == rows and o.shape == v.shape
            and g.shape == (rows, v.shape[1]) and beta.shape == g.shape
            and src_slot.shape[0] == rows and (dst_slot is None or dst_slot.shape[0] == rows)
            and state.shape[1:] == (v.shape[1], v.shape[2], q.shape[2])):
        raise ValueError("inconsistent decode shapes")
    d = _dims(q, v, scale)
    args = (ctypes.byref(d), rows, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
            state.shape[0], _ptr(src_slot), _ptr(dst_slot), _ptr(o), _ptr(dev_status), _stream(stream))
    keep = (d, q, k, v, g, beta, state, src_slot, dst_slot, o, dev_status)
    return _PreparedCall(lib.gdn_decode_packed, args, "gdn_decode_packed", keep)


def gdn_prep_inputs(q_raw, k_raw, a, b, A_log, dt_bias, q, k, g, beta, eps: float = 1e-6,
                    stream=None) -> None:
    """Input preparation: normalised q, k (bf16) and g, beta (fp32) from raw
    projections (see gdn.h).  q, k may alias q_raw, k_raw."""
    lib = load_library()
    bf, f32 = torch.bfloat16, torch.float32
    q_raw, k_raw = _dev(q_raw, "q_raw", bf, 3), _dev(k_raw, "k_raw", bf, 3)
    q, k = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3)
    a, b, g, beta = (_dev(x, n, f32, 2) for x, n in ((a, "a"), (b, "b"), (g, "g"), (beta, "beta")))
    A_log, dt_bias = _dev(A_log, "A_log", f32, 1), _dev(dt_bias, "dt_bias", f32, 1)
    T, h_v = a.shape
    if not (k_raw.shape == q_raw.shape == q.shape == k.shape and q.shape[0] == T and b.shape == a.shape
            and g.shape == a.shape and beta.shape == a.shape and A_log.shape == (h_v,)
            and dt_bias.shape == (h_v,)):
        raise ValueError("inconsistent input-preparation shapes")
    d = Dims(q.shape[1], h_v, q.shape[2], q.shape[2], 1.0)
    _check(lib.gdn_prep_inputs(ctypes.byref(d), T, _ptr(q_raw), _ptr(k_raw), _ptr(a), _ptr(b), _ptr(A_log),
                               _ptr(dt_bias), float(eps), _ptr(q), _ptr(k), _ptr(g), _ptr(beta),
                               _stream(stream)),
           "gdn_prep_inputs")


def gdn_decode_packed_raw(q_raw, k_raw, v, a, b, A_log, dt_bias, state, src_slot, o, dst_slot=None,
                          dev_status=None, eps: float = 1e-6, scale: float = 1.0, stream=None) -> None:
    """Packed decode with the input preparation fused in (see gdn.h)."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q_raw, k_raw, v = _dev(q_raw, "q_raw", bf, 3), _dev(k_raw, "k_raw", bf, 3), _dev(v, "v", bf, 3)
    a, b = _dev(a, "a", f32, 2), _dev(b, "b", f32, 2)
    A_log, dt_bias = _dev(A_log, "A_log", f32, 1), _dev(dt_bias, "dt_bias", f32, 1)
    state = _dev(state, "state", f32, 4)
    src_slot = _dev(src_slot, "src_slot", i32, 1)
    dst_slot = _dev(dst_slot, "dst_slot", i32, 1, optional=True)
    o = _dev(o, "o", bf, 3)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    rows = q_raw.shape[0]
    if not (k_raw.shape == q_raw.shape and v.shape[0] == rows and o.shape == v.shape
            and a.shape == (rows, v.shape[1]) and b.shape == a.shape
            and A_log.shape == (v.shape[1],) and dt_bias.shape == A_log.shape
            and src_slot.shape[0] == rows and (dst_slot is None or dst_slot.shape[0] == rows)
            and state.shape[1:] == (v.shape[1], v.shape[2], q_raw.shape[2])):
        raise ValueError("inconsistent decode shapes")
    d = _dims(q_raw, v, scale)
    _check(lib.gdn_decode_packed_raw(ctypes.byref(d), rows, _ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a),
                                     _ptr(b), _ptr(A_log), _ptr(dt_bias), float(eps), _ptr(state),
                                     state.shape[0], _ptr(src_slot), _ptr(dst_slot), _ptr(o),
                                     _ptr(dev_status), _stream(stream)),
           "gdn_decode_packed_raw")


def gdn_decode_multi(tokens_per_row: int, q, k, v, g, beta, state, src_slot, o, dst_slots=None,
                     dev_status=None, scale: float = 1.0, stream=None) -> None:
    """Multi-token decode: ``q.shape[0] // tokens_per_row`` rows of
    ``tokens_per_row`` consecutive tokens each (see gdn.h)."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    state = _dev(state, "state", f32, 4)
    src_slot = _dev(src_slot, "src_slot", i32, 1)
    dst_slots = _dev(dst_slots, "dst_slots", i32, 1, optional=True)
    o = _dev(o, "o", bf, 3)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    T = int(tokens_per_row)
    ntok = q.shape[0]
    if T < 1 or ntok % T:
        raise ValueError("q.shape[0] must be a multiple of tokens_per_row >= 1")
    rows = ntok // T
    if not (k.shape == q.shape and v.shape[0] == ntok and o.shape == v.shape
            and g.shape == (ntok, v.shape[1]) and beta.shape == g.shape
            and src_slot.shape[0] == rows and (dst_slots is None or dst_slots.shape[0] == ntok)
            and state.shape[1:] == (v.shape[1], v.shape[2], q.shape[2])):
        raise ValueError("inconsistent multi-token decode shapes")
    d = _dims(q, v, scale)
    _check(lib.gdn_decode_multi(ctypes.byref(d), rows, T, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(state), state.shape[0], _ptr(src_slot),
                                _ptr(dst_slots), _ptr(o), _ptr(dev_status), _stream(stream)),
           "gdn_decode_multi")


def gdn_prefill_varlen(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, o, state=None,
                       src_slot=None, dst_slot=None, chunk_states=None, emit_every_chunks: int = 0,
                       dev_status=None, scale: float = 1.0, stream=None, workspace=None) -> None:
    """Chunked varlen prefill (see gdn.h).  ``cu_seqlens_host`` is a host
    sequence (list or CPU tensor) with the same values as ``cu_seqlens``;
    ``workspace`` an optional uint8 device tensor (see
    ``gdn_prefill_workspace_bytes``)."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    o = _dev(o, "o", bf, 3)
    cu_seqlens = _dev(cu_seqlens, "cu_seqlens", i32, 1)
    state = _dev(state, "state", f32, 4, optional=True)
    src_slot = _dev(src_slot, "src_slot", i32, 1, optional=True)
    dst_slot = _dev(dst_slot, "dst_slot", i32, 1, optional=True)
    chunk_states = _dev(chunk_states, "chunk_states", f32, 4, optional=True)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    keep, cu_h = _host_i32(cu_seqlens_host, "cu_seqlens_host")
    n = cu_seqlens.shape[0] - 1
    if len(keep) != n + 1:
        raise ValueError("cu_seqlens_host must have num_seqs + 1 entries")
    T = q.shape[0]
    if not (k.shape == q.shape and v.shape[0] == T and o.shape == v.shape
            and g.shape == (T, v.shape[1]) and beta.shape == g.shape):
        raise ValueError("inconsistent prefill shapes")
    d = _dims(q, v, scale)
    cap = 0 if chunk_states is None else chunk_states.shape[0]
    ws, ws_bytes = _workspace(workspace, d, n, T)
    _check(lib.gdn_prefill_varlen(ctypes.byref(d), n, _ptr(cu_seqlens), cu_h, _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                  0 if state is None else state.shape[0], _ptr(src_slot),
                                  _ptr(dst_slot), _ptr(o), _ptr(chunk_states),
                                  int(emit_every_chunks), cap, ws, ws_bytes, _ptr(dev_status),
                                  _stream(stream)),
           "gdn_prefill_varlen")


def gdn_prefill_varlen_apc(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, o, state, block_table,
                           block_first, emit_every_chunks: int, src_slot=None, dst_slot=None,
                           dev_status=None, scale: float = 1.0, stream=None, workspace=None) -> None:
    """Chunked varlen prefill emitting into cache blocks: ``block_table``
    int32 [num_seqs][max_blocks], ``block_first`` int32 [num_seqs] (see gdn.h)."""
    lib = load_library()
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    o = _dev(o, "o", bf, 3)
    cu_seqlens = _dev(cu_seqlens, "cu_seqlens", i32, 1)
    state = _dev(state, "state", f32, 4)
    block_table = _dev(block_table, "block_table", i32, 2)
    block_first = _dev(block_first, "block_first", i32, 1)
    src_slot = _dev(src_slot, "src_slot", i32, 1, optional=True)
    dst_slot = _dev(dst_slot, "dst_slot", i32, 1, optional=True)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    keep, cu_h = _host_i32(cu_seqlens_host, "cu_seqlens_host")
    n = cu_seqlens.shape[0] - 1
    if len(keep) != n + 1 or block_table.shape[0] != n or block_first.shape[0] != n:
        raise ValueError("cu_seqlens_host, block_table and block_first must cover num_seqs sequences")
    T = q.shape[0]
    if not (k.shape == q.shape and v.shape[0] == T and o.shape == v.shape
            and g.shape == (T, v.shape[1]) and beta.shape == g.shape):
        raise ValueError("inconsistent prefill shapes")
    d = _dims(q, v, scale)
    ws, ws_bytes = _workspace(workspace, d, n, T)
    _check(lib.gdn_prefill_varlen_apc(ctypes.byref(d), n, _ptr(cu_seqlens), cu_h, _ptr(q), _ptr(k),
                                      _ptr(v), _ptr(g), _ptr(beta), _ptr(state), state.shape[0],
                                      _ptr(src_slot), _ptr(dst_slot), _ptr(o), int(emit_every_chunks),
                                      _ptr(block_table), block_table.shape[1], _ptr(block_first),
                                      ws, ws_bytes, _ptr(dev_status), _stream(stream)),
           "gdn_prefill_varlen_apc")


def _mixed_args(num_decodes, q, k, v, g, beta, cu_seqlens_p, cu_seqlens_p_host, state, dec_src_slot, o,
                dec_dst_slot, pre_src_slot, pre_dst_slot, chunk_states, emit_every_chunks, dev_status,
                scale, stream, workspace):
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = _dev(q, "q", bf, 3), _dev(k, "k", bf, 3), _dev(v, "v", bf, 3)
    g, beta = _dev(g, "g", f32, 2), _dev(beta, "beta", f32, 2)
    o = _dev(o, "o", bf, 3)
    state = _dev(state, "state", f32, 4)
    dec_src_slot = _dev(dec_src_slot, "dec_src_slot", i32, 1, optional=num_decodes == 0)
    dec_dst_slot = _dev(dec_dst_slot, "dec_dst_slot", i32, 1, optional=True)
    pre_src_slot = _dev(pre_src_slot, "pre_src_slot", i32, 1, optional=True)
    pre_dst_slot = _dev(pre_dst_slot, "pre_dst_slot", i32, 1, optional=True)
    chunk_states = _dev(chunk_states, "chunk_states", f32, 4, optional=True)
    dev_status = _dev(dev_status, "dev_status", i32, optional=True)
    cu_seqlens_p = _dev(cu_seqlens_p, "cu_seqlens_p", i32, 1, optional=True)
    n_p = 0 if cu_seqlens_p is None else cu_seqlens_p.shape[0] - 1
    keep, cu_h = _host_i32(cu_seqlens_p_host if cu_seqlens_p_host is not None else [0], "cu_seqlens_p_host")
    if n_p and len(keep) != n_p + 1:
        raise ValueError("cu_seqlens_p_host must have num_prefills + 1 entries")
    T = q.shape[0]
    if not (k.shape == q.shape and v.shape[0] == T and o.shape == v.shape
            and g.shape == (T, v.shape[1]) and beta.shape == g.shape):
        raise ValueError("inconsistent mixed-step shapes")
    if n_p and int(keep[-1]) + num_decodes != T:
        raise ValueError("token count does not match num_decodes + cu_seqlens_p_host[-1]")
    d = _dims(q, v, scale)
    cap = 0 if chunk_states is None else chunk_states.shape[0]
    ws, ws_bytes = _workspace(workspace, d, n_p, T - int(num_decodes))
    # `keep` and `d` hold the memory that cu_h and byref(d) point into.
    return (keep, d), [ctypes.byref(d), int(num_decodes), n_p, _ptr(cu_seqlens_p), cu_h,
                       _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                       state.shape[0], _ptr(dec_src_slot), _ptr(dec_dst_slot),
                       _ptr(pre_src_slot), _ptr(pre_dst_slot), _ptr(o), _ptr(chunk_states),
                       int(emit_every_chunks), cap, ws, ws_bytes, _ptr(dev_status), _stream(stream)]


def gdn_mixed_step(num_decodes: int, q, k, v, g, beta, cu_seqlens_p, cu_seqlens_p_host, state,
                   dec_src_slot, o, dec_dst_slot=None, pre_src_slot=None, pre_dst_slot=None,
                   chunk_states=None, emit_every_chunks: int = 0, dev_status=None,
                   scale: float = 1.0, stream=None, workspace=None) -> None:
    """Mixed step: decode rows [0, num_decodes) then prefill sequences."""
    lib = load_library()
    _keep, args = _mixed_args(num_decodes, q, k, v, g, beta, cu_seqlens_p, cu_seqlens_p_host, state,
                              dec_src_slot, o, dec_dst_slot, pre_src_slot, pre_dst_slot, chunk_states,
                              emit_every_chunks, dev_status, scale, stream, workspace)
    _check(lib.gdn_mixed_step(*args), "gdn_mixed_step")


def _event_handle(ev, stream):
    # torch creates the CUDA event on its first record; recording it once on
    # `stream` here is harmless because the library records it again.
    if ev.cuda_event == 0:
        ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ctypes.c_void_p(ev.cuda_event)


def gdn_mixed_step_colaunch(num_decodes: int, q, k, v, g, beta, cu_seqlens_p, cu_seqlens_p_host, state,
                            dec_src_slot, o, aux_stream, fork_event, join_event, dec_dst_slot=None,
                            pre_src_slot=None, pre_dst_slot=None, chunk_states=None,
                            emit_every_chunks: int = 0, dev_status=None, scale: float = 1.0,
                            stream=None, workspace=None) -> None:
    """Mixed step with the decode rows on `aux_stream` (a torch.cuda.Stream)
    running beside the prefill on `stream`; `fork_event` and `join_event` are
    torch.cuda.Event objects the call records (fork on `stream`, join on
    `aux_stream`).  The decode and prefill slots must not overlap."""
    lib = load_library()
    _keep, args = _mixed_args(num_decodes, q, k, v, g, beta, cu_seqlens_p, cu_seqlens_p_host, state,
                              dec_src_slot, o, dec_dst_slot, pre_src_slot, pre_dst_slot, chunk_states,
                              emit_every_chunks, dev_status, scale, stream, workspace)
    if aux_stream is None:
        extra = [None, None, None]
    else:
        extra = [ctypes.c_void_p(aux_stream.cuda_stream), _event_handle(fork_event, stream),
                 _event_handle(join_event, stream)]
    _check(lib.gdn_mixed_step_colaunch(*args, *extra), "gdn_mixed_step_colaunch")


# ---------------------------------------------------------------------------
# host-only helpers
# ---------------------------------------------------------------------------

def gdn_prefill_num_emits(cu_seqlens_host, emit_every_chunks: int) -> int:
    keep, p = _host_i32(cu_seqlens_host, "cu_seqlens_host")
    n = load_library().gdn_prefill_num_emits(p, len(keep) - 1, int(emit_every_chunks))
    if n < 0:
        raise ValueError("invalid cu_seqlens_host")
    return int(n)


def gdn_prefill_emit_offsets(cu_seqlens_host, emit_every_chunks: int) -> list[int]:
    keep, p = _host_i32(cu_seqlens_host, "cu_seqlens_host")
    out = (ctypes.c_int64 * len(keep))()
    _check(load_library().gdn_prefill_emit_offsets(p, len(keep) - 1, int(emit_every_chunks),
                                                   ctypes.cast(out, ctypes.c_void_p)),
           "gdn_prefill_emit_offsets")
    return [int(x) for x in out]


def gdn_align_block_size(block_size: int) -> int:
    return int(load_library().gdn_align_block_size(int(block_size)))


def gdn_floor_prefix_hit(hit_tokens: int, prompt_tokens: int, block_size: int) -> int:
    return int(load_library().gdn_floor_prefix_hit(int(hit_tokens), int(prompt_tokens), int(block_size)))


def gdn_grid_emit_every_chunks(block_size: int) -> int:
    return int(load_library().gdn_grid_emit_every_chunks(int(block_size)))


def gdn_prefill_workspace_bytes(h_k: int, h_v: int, d: int, num_seqs: int, total_tokens: int) -> int:
    """Device scratch (bytes) a prefill of ``num_seqs`` sequences needs."""
    dims = Dims(int(h_k), int(h_v), int(d), int(d), 1.0)
    n = load_library().gdn_prefill_workspace_bytes(ctypes.byref(dims), int(num_seqs), int(total_tokens))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid prefill dims or sizes")
    return int(n)


def gdn_status_from_device(word: int) -> int:
    """Status of a finished call from the device status word it wrote."""
    return int(load_library().gdn_status_from_device(int(word)))


def gdn_status_string(status: int) -> str:
    return load_library().gdn_status_string(int(status)).decode()
