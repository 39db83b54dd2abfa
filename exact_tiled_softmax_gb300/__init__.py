"""exact_tiled_softmax_gb300: exact masked attention on one GB300 (sm_103a).

A thin ctypes binding over ``libexattn.so`` (C ABI in ``include/exattn.h``).
Every step of the forward and reverse pass runs in the library's CUDA
kernels; this module only checks tensors, allocates outputs and workspaces
with torch (device memory and streams are all torch is used for) and passes
raw pointers.  There is no CPU fallback: if the library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["fwd", "bwd", "fwd_workspace_size", "bwd_workspace_size", "device_status",
           "set_path", "library_path", "load_library", "ExattnError", "Shape",
           "record_kernel_events", "launch_count", "workspace", "bwd_noalloc",
           "noalloc_device_status",
           "fwd_splitkv", "QKShape",
           "MASK_NONE", "MASK_CAUSAL", "MASK_WINDOW", "MASK_BITMASK"]

MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BITMASK = 0, 1, 2, 3
_MASKS = {"none": MASK_NONE, "causal": MASK_CAUSAL, "window": MASK_WINDOW,
          "bitmask": MASK_BITMASK}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}
_PATHS = {"auto": 0, "simt": 1, "atomic_dq": 2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


def library_path() -> str:
    return os.path.join(_HERE, "libexattn.so")


class ExattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = load_library()
        msg = lib.exattn_status_string(status).decode()
        detail = lib.exattn_last_error().decode()
        super().__init__(f"{where}: status {status} ({msg})" + (f": {detail}" if detail else ""))


class QKShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("nq", ctypes.c_int),
                ("nk", ctypes.c_int), ("d", ctypes.c_int), ("v", ctypes.c_int),
                ("dtype", ctypes.c_int)]


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("n", ctypes.c_int),
                ("d", ctypes.c_int), ("v", ctypes.c_int), ("dtype", ctypes.c_int)]


def load_library():
    """Load libexattn.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libexattn.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, sz, ci, cf = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    sp = ctypes.POINTER(Shape)
    lib.exattn_set_path.argtypes = [ci]
    lib.exattn_set_path.restype = ci
    lib.exattn_fwd_workspace_size.argtypes = [sp, ci]
    lib.exattn_fwd_workspace_size.restype = sz
    lib.exattn_bwd_workspace_size.argtypes = [sp, ci]
    lib.exattn_bwd_workspace_size.restype = sz
    lib.attn_fwd.argtypes = [sp, vp, vp, vp, cf, ci, ci, vp, vp, vp, vp, sz, vp]
    lib.attn_fwd.restype = ci
    lib.attn_bwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, cf, ci, ci, vp, vp, vp, vp, vp, sz, vp]
    lib.attn_bwd.restype = ci
    u64 = ctypes.c_uint64
    lib.attn_fwd_dropout.argtypes = [sp, vp, vp, vp, cf, ci, ci, vp, cf, u64, vp, vp, vp, sz, vp]
    lib.attn_fwd_dropout.restype = ci
    lib.attn_bwd_dropout.argtypes = [sp, vp, vp, vp, vp, vp, vp, cf, ci, ci, vp, cf, u64, vp, vp,
                                     vp, vp, sz, vp]
    lib.attn_bwd_dropout.restype = ci
    qsp = ctypes.POINTER(QKShape)
    lib.exattn_fwd_qk_workspace_size.argtypes = [qsp, ci]
    lib.exattn_fwd_qk_workspace_size.restype = sz
    lib.exattn_bwd_qk_workspace_size.argtypes = [qsp, ci]
    lib.exattn_bwd_qk_workspace_size.restype = sz
    lib.attn_fwd_qk.argtypes = [qsp, vp, vp, vp, cf, ci, ci, vp, cf, u64, vp, vp, vp, sz, vp]
    lib.attn_fwd_qk.restype = ci
    lib.attn_bwd_qk.argtypes = [qsp, vp, vp, vp, vp, vp, vp, cf, ci, ci, vp, cf, u64, vp, vp, vp,
                                vp, sz, vp]
    lib.attn_bwd_qk.restype = ci
    lib.exattn_device_status.argtypes = [vp, vp]
    lib.exattn_device_status.restype = ci
    lib.exattn_status_string.argtypes = [ci]
    lib.exattn_status_string.restype = ctypes.c_char_p
    lib.exattn_record_kernel_events.argtypes = [ci, vp, vp]
    lib.exattn_record_kernel_events.restype = ci
    lib.exattn_launch_count.argtypes = []
    lib.exattn_launch_count.restype = ctypes.c_ulonglong
    lib.attn_bwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, cf, ci, ci, vp, vp, vp, vp, vp]
    lib.attn_bwd_noalloc.restype = ci
    lib.exattn_noalloc_device_status.argtypes = [vp]
    lib.exattn_noalloc_device_status.restype = ci
    lib.exattn_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint, vp]
    lib.exattn_selftest_wait_timeout.restype = ci
    qp = ctypes.POINTER(QKShape)
    lib.exattn_splitkv_workspace_size.argtypes = [qp, ci]
    lib.exattn_splitkv_workspace_size.restype = sz
    lib.attn_fwd_splitkv.argtypes = [qp, vp, vp, vp, cf, ci, ci, vp, ci, vp, vp, vp, sz, vp]
    lib.attn_fwd_splitkv.restype = ci
    lib.exattn_last_error.argtypes = []
    lib.exattn_last_error.restype = ctypes.c_char_p
    lib.exattn_host_step_workspace_size.argtypes = [sp, ci]
    lib.exattn_host_step_workspace_size.restype = sz
    lib.attn_step_host.argtypes = [sp, vp, vp, vp, vp, cf, ci, ci, vp, vp, vp, vp, vp, vp, vp, sz,
                                   vp]
    lib.attn_step_host.restype = ci
    _lib = lib
    return lib


def set_path(path: str) -> str:
    """Process-wide kernel path: "auto" (tensor-core kernels where supported), "simt",
    or "atomic_dq" (auto, with the fp32-atomic dQ form of the reverse pass)."""
    prev = load_library().exattn_set_path(_PATHS[path])
    return {v: k for k, v in _PATHS.items()}[prev]


def _mask_kind(mask) -> int:
    return _MASKS[mask] if isinstance(mask, str) else int(mask)


def _shape(q: torch.Tensor, v: torch.Tensor) -> Shape:
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [batch, heads, n, width] tensors")
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, n, d = q.shape
    return Shape(B, H, n, d, v.shape[-1], _DTYPES[q.dtype])


def fwd_workspace_size(shape: Shape, mask) -> int:
    return load_library().exattn_fwd_workspace_size(ctypes.byref(shape), _mask_kind(mask))


def bwd_workspace_size(shape: Shape, mask) -> int:
    return load_library().exattn_bwd_workspace_size(ctypes.byref(shape), _mask_kind(mask))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(ts, dtype, device):
    for t in ts:
        if t is None:
            continue
        if t.device != device or not t.is_contiguous():
            raise ValueError("tensors must be contiguous and on the same CUDA device")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"dtype mismatch: {t.dtype} vs {dtype}")


def _check_shapes(q, k, v, y=None, dy=None, L=None, dq=None, dk=None, dv=None, same_n=False):
    """Shapes agree with q [B,H,nq,d], k [B,H,nk,d], v [B,H,nk,v]: Y and dY are
    [B,H,nq,v], L fp32 [B,H,nq], dQ/dK/dV like Q/K/V.  Raises ValueError before
    anything reaches the library, which trusts the sizes it is given."""
    for name, t, nd in (("q", q, 4), ("k", k, 4), ("v", v, 4), ("y", y, 4), ("dy", dy, 4),
                        ("L", L, 3), ("dq", dq, 4), ("dk", dk, 4), ("dv", dv, 4)):
        if t is not None and t.dim() != nd:
            raise ValueError(f"{name} must have {nd} dimensions, got shape {tuple(t.shape)}")
    B, H, nq, d = q.shape
    nk, vw = k.shape[2], v.shape[3]
    want = {"k": (B, H, nk, d), "v": (B, H, nk, vw), "y": (B, H, nq, vw),
            "dy": (B, H, nq, vw), "L": (B, H, nq), "dq": (B, H, nq, d), "dk": (B, H, nk, d),
            "dv": (B, H, nk, vw)}
    for name, t in (("k", k), ("v", v), ("y", y), ("dy", dy), ("L", L), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if t is not None and tuple(t.shape) != want[name]:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {want[name]}")
    if same_n and nk != nq:
        raise ValueError(f"k and v must have q's sequence length {nq}, got {nk}")
    if L is not None:
        if L.dtype != torch.float32 or not L.is_contiguous() or L.device != q.device:
            raise ValueError("L must be a contiguous float32 tensor on q's device")


_WORD_DTYPES = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _check_aux(q, nk, kind, bitmask=None, ws=None, bitmask_device=None):
    """The bitmask and the workspace, which the library takes as bare pointers:
    the bitmask must be 32-bit words, contiguous, on ``bitmask_device`` (default:
    q's device) and, for the bitmask mask kind, hold at least nq * ceil(nk / 32)
    words (the kernels read that many); the workspace must be contiguous and on
    q's device.  Raises ValueError before anything reaches the library."""
    if bitmask is not None:
        dev = q.device if bitmask_device is None else bitmask_device
        if (bitmask.dtype not in _WORD_DTYPES or not bitmask.is_contiguous()
                or bitmask.device != dev):
            raise ValueError(f"bitmask must be contiguous 32-bit words on {dev}")
        need = q.shape[2] * ((nk + 31) // 32)
        if kind == MASK_BITMASK and bitmask.numel() < need:
            raise ValueError(f"bitmask holds {bitmask.numel()} words, the mask needs {need}")
    if ws is not None and (ws.device != q.device or not ws.is_contiguous()):
        raise ValueError("the workspace must be a contiguous tensor on q's device")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned device byte buffer of at least ``nbytes``."""
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _qk_shape(q, k, v) -> QKShape:
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [batch, heads, n, width] tensors")
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, nq, d = q.shape
    return QKShape(B, H, nq, k.shape[2], d, v.shape[-1], _DTYPES[q.dtype])


def _fwd_qk(lib, q, k, v, scale, kind, window, bitmask, y, L, ws, stream, dropout_p, seed):
    shape = _qk_shape(q, k, v)
    if y is None:
        y = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if L is None:
        L = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(lib.exattn_fwd_qk_workspace_size(ctypes.byref(shape), kind), q.device)
    st = lib.attn_fwd_qk(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale), kind,
                         int(window), _ptr(bitmask), float(dropout_p), int(seed), _ptr(y),
                         _ptr(L), _ptr(ws), _nbytes(ws), _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_fwd_qk")
    return y, L


def _bwd_qk(lib, q, k, v, y, dy, L, scale, kind, window, bitmask, dq, dk, dv, ws, stream,
            dropout_p, seed):
    shape = _qk_shape(q, k, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if ws is None:
        ws = workspace(lib.exattn_bwd_qk_workspace_size(ctypes.byref(shape), kind), q.device)
    st = lib.attn_bwd_qk(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(dy),
                         _ptr(L), float(scale), kind, int(window), _ptr(bitmask),
                         float(dropout_p), int(seed), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                         _nbytes(ws), _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_bwd_qk")
    return dq, dk, dv


def fwd(q, k, v, scale, mask="none", window=0, bitmask=None, y=None, L=None, ws=None,
        stream=None, dropout_p=0.0, seed=0):
    """Forward pass -> (Y, L).  q [B,H,nq,d], k [B,H,nk,d], v [B,H,nk,v]; bitmask
    int32/uint32 words.  nq != nk runs attn_fwd_qk (queries aligned to the end of
    the keys).  ``dropout_p`` > 0 drops probabilities with the replayable mask of
    ``seed``; the reverse pass must get the same two values."""
    lib = load_library()
    _check((q, k, v, y), q.dtype, q.device)
    _check_shapes(q, k, v, y=y, L=L)
    kind = _mask_kind(mask)
    _check_aux(q, k.shape[2], kind, bitmask, ws)
    if k.shape[2] != q.shape[2]:
        return _fwd_qk(lib, q, k, v, scale, kind, window, bitmask, y, L, ws, stream, dropout_p,
                       seed)
    shape = _shape(q, v)
    if y is None:
        y = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if L is None:
        L = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    need = lib.exattn_fwd_workspace_size(ctypes.byref(shape), kind)
    if ws is None:
        ws = workspace(need, q.device)
    if dropout_p:
        st = lib.attn_fwd_dropout(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale),
                                  kind, int(window), _ptr(bitmask), float(dropout_p), int(seed),
                                  _ptr(y), _ptr(L), _ptr(ws), _nbytes(ws), _stream(stream))
    else:
        st = lib.attn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale), kind,
                          int(window), _ptr(bitmask), _ptr(y), _ptr(L), _ptr(ws), _nbytes(ws),
                          _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_fwd_dropout" if dropout_p else "attn_fwd")
    return y, L


def bwd(q, k, v, y, dy, L, scale, mask="none", window=0, bitmask=None, dq=None, dk=None,
        dv=None, ws=None, stream=None, dropout_p=0.0, seed=0):
    """Reverse pass -> (dQ, dK, dV) for the upstream gradient dy (with the forward
    pass's ``dropout_p`` and ``seed`` when it used dropout)."""
    lib = load_library()
    _check((q, k, v, y, dy, dq, dk, dv), q.dtype, q.device)
    _check_shapes(q, k, v, y=y, dy=dy, L=L, dq=dq, dk=dk, dv=dv)
    kind = _mask_kind(mask)
    _check_aux(q, k.shape[2], kind, bitmask, ws)
    if k.shape[2] != q.shape[2]:
        return _bwd_qk(lib, q, k, v, y, dy, L, scale, kind, window, bitmask, dq, dk, dv, ws,
                       stream, dropout_p, seed)
    shape = _shape(q, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = lib.exattn_bwd_workspace_size(ctypes.byref(shape), kind)
    if ws is None:
        ws = workspace(need, q.device)
    if dropout_p:
        st = lib.attn_bwd_dropout(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(y),
                                  _ptr(dy), _ptr(L), float(scale), kind, int(window),
                                  _ptr(bitmask), float(dropout_p), int(seed), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(ws), _nbytes(ws), _stream(stream))
    else:
        st = lib.attn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(dy),
                          _ptr(L), float(scale), kind, int(window), _ptr(bitmask), _ptr(dq),
                          _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws), _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_bwd")
    return dq, dk, dv


def fwd_splitkv(q, k, v, scale, mask="none", window=0, bitmask=None, num_splits=0, y=None,
                L=None, ws=None, stream=None):
    """Split-KV forward -> (Y, L) for q [B,H,nq,d] against k [B,H,nk,d], v [B,H,nk,v];
    the queries are the last nq positions of the key sequence.  ``num_splits``
    0 lets the library choose the number of key chunks."""
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [batch, heads, n, width] tensors")
    _check((q, k, v, y), q.dtype, q.device)
    _check_shapes(q, k, v, y=y, L=L)
    B, H, nq, d = q.shape
    shape = QKShape(B, H, nq, k.shape[2], d, v.shape[-1], _DTYPES[q.dtype])
    kind = _mask_kind(mask)
    _check_aux(q, k.shape[2], kind, bitmask, ws)
    if y is None:
        y = torch.empty((B, H, nq, v.shape[-1]), dtype=q.dtype, device=q.device)
    if L is None:
        L = torch.empty((B, H, nq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(lib.exattn_splitkv_workspace_size(ctypes.byref(shape), int(num_splits)),
                       q.device)
    st = lib.attn_fwd_splitkv(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale), kind,
                              int(window), _ptr(bitmask), int(num_splits), _ptr(y), _ptr(L),
                              _ptr(ws), _nbytes(ws), _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_fwd_splitkv")
    return y, L


def bwd_noalloc(q, k, v, y, dy, L, scale, mask="none", window=0, bitmask=None, dq=None,
                dk=None, dv=None, stream=None, check_status=False):
    """Reverse pass through attn_bwd_noalloc: no workspace is passed or allocated;
    the library's own 64 MiB scratch array is used instead.  With
    ``check_status`` the call then synchronises the stream and raises
    ExattnError if the kernels recorded a condition (an empty allowed set or a
    bounded wait that gave up) in the scratch array's status word."""
    lib = load_library()
    _check((q, k, v, y, dy, dq, dk, dv), q.dtype, q.device)
    _check_shapes(q, k, v, y=y, dy=dy, L=L, dq=dq, dk=dk, dv=dv, same_n=True)
    _check_aux(q, k.shape[2], _mask_kind(mask), bitmask)
    shape = _shape(q, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = lib.attn_bwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(y),
                              _ptr(dy), _ptr(L), float(scale), _mask_kind(mask), int(window),
                              _ptr(bitmask), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream))
    if st != 0:
        raise ExattnError(st, "attn_bwd_noalloc")
    if check_status:
        st = noalloc_device_status(stream)
        if st != 0:
            raise ExattnError(st, "attn_bwd_noalloc (device status)")
    return dq, dk, dv


def noalloc_device_status(stream=None) -> int:
    """exattn_noalloc_device_status: synchronise the stream, then read the status
    word that the last attn_bwd_noalloc call left in the library's scratch array."""
    return load_library().exattn_noalloc_device_status(_stream(stream))


KERNEL_FWD, KERNEL_DELTA, KERNEL_BWD, KERNEL_DQ_CONVERT, KERNEL_BWD_Q = 0, 1, 2, 3, 4
KERNEL_SPLIT_PARTIAL, KERNEL_SPLIT_MERGE, KERNEL_SPLIT32 = 5, 6, 7


def step_host(q, k, v, dy, scale, mask="none", window=0, bitmask=None, out=None, ws=None,
              stream=None, device=None):
    """attn_step_host: forward and reverse pass on CPU tensors (pinned for
    asynchronous copies) -> (Y, L, dQ, dK, dV), CPU tensors.  ``out`` may give
    the five outputs (pinned, to be reused); ``ws`` a device workspace of
    exattn_host_step_workspace_size bytes.  Returns once the step is queued:
    synchronise ``stream`` (default: the current stream of ``device``) before
    reading the outputs."""
    lib = load_library()
    dev = torch.device("cuda") if device is None else torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    for t in (q, k, v, dy):
        if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("step_host takes contiguous CPU tensors of one dtype")
    _check_shapes(q, k, v, dy=dy, same_n=True)
    kind = _mask_kind(mask)
    _check_aux(q, k.shape[2], kind, bitmask, bitmask_device=torch.device("cpu"))
    if ws is not None and (ws.device != dev or not ws.is_contiguous()):
        raise ValueError("the workspace must be a contiguous tensor on the step's device")
    shape = _shape(q, v)
    if out is None:
        pin = torch.cuda.is_available()
        out = (torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, pin_memory=pin),
               torch.empty(q.shape[:-1], dtype=torch.float32, pin_memory=pin),
               torch.empty(q.shape, dtype=q.dtype, pin_memory=pin),
               torch.empty(k.shape, dtype=q.dtype, pin_memory=pin),
               torch.empty(v.shape, dtype=q.dtype, pin_memory=pin))
    y, L, dq, dk, dv = out
    rows = tuple(q.shape[:-1])
    want = {"y": (rows + (v.shape[-1],), q.dtype), "L": (rows, torch.float32),
            "dq": (tuple(q.shape), q.dtype), "dk": (tuple(k.shape), q.dtype),
            "dv": (tuple(v.shape), q.dtype)}
    for name, t in zip(("y", "L", "dq", "dk", "dv"), out):
        if ((tuple(t.shape), t.dtype) != want[name] or t.device.type != "cpu"
                or not t.is_contiguous()):
            raise ValueError(f"out {name} must be a contiguous CPU tensor of shape "
                             f"{want[name][0]} and dtype {want[name][1]}")
    need = lib.exattn_host_step_workspace_size(ctypes.byref(shape), kind)
    if ws is None:
        ws = workspace(need, dev)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    st = lib.attn_step_host(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), float(scale),
                            kind, int(window), _ptr(bitmask), _ptr(y), _ptr(L), _ptr(dq), _ptr(dk),
                            _ptr(dv), _ptr(ws), _nbytes(ws), ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise ExattnError(st, "attn_step_host")
    return y, L, dq, dk, dv


def record_kernel_events(which: int, start, stop) -> None:
    """One-shot: record torch.cuda.Event ``start``/``stop`` around the next launch
    of kernel ``which`` (one of the KERNEL_* roles)."""
    for e in (start, stop):
        if e.cuda_event == 0:
            raise ValueError("events must be created (record or query them once) first")
    if load_library().exattn_record_kernel_events(which, ctypes.c_void_p(start.cuda_event),
                                                  ctypes.c_void_p(stop.cuda_event)) != 0:
        raise ValueError(f"unknown kernel {which}")


def launch_count() -> int:
    """Kernels launched by the library since it was loaded."""
    return int(load_library().exattn_launch_count())


def device_status(ws, stream=None) -> int:
    """Synchronise the stream and read the status word of workspace ``ws``."""
    return load_library().exattn_device_status(_ptr(ws), _stream(stream))
