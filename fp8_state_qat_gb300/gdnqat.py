"""ctypes binding of libgdnqat.so (include/gdnqat.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels. torch supplies device memory (outputs are allocated here when not given) and the
current CUDA stream. There is no fallback: if the library is missing or the device is not
sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED_ARCH = 2
GDN_ERR_UNSUPPORTED_SHAPE = 3
GDN_ERR_WORKSPACE_TOO_SMALL = 4
GDN_ERR_CUDA = 5
GDN_ERR_DEVICE_TIMEOUT = 6

GDN_FLAG_STATE_QDQ = 1
GDN_FLAG_W_QDQ = 2
GDN_FLAG_KDA = 4
GDN_FLAG_STATE_INT8 = 8

# every extern "C" symbol of include/gdnqat.h
EXPORTED = ("gdn_chunk_fwd_workspace_size", "gdn_chunk_fwd", "gdn_chunk_fwd_noalloc",
            "kda_chunk_fwd_workspace_size", "kda_chunk_fwd",
            "gdn_prefill_decode_workspace_size", "gdn_prefill_decode_fwd",
            "gdn_chunk_bwd_workspace_size", "gdn_chunk_bwd", "kda_chunk_bwd_workspace_size", "kda_chunk_bwd",
            "kda_prefill_decode_workspace_size", "kda_prefill_decode_fwd",
            "gdn_decode_step", "fp8_tile_qdq", "int8_block_qdq", "gdn_status_string", "gdn_check_device_status")


class GdnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class ChunkArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_host", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("hT", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("N", ctypes.c_int32), ("Hqk", ctypes.c_int32),
                ("Hv", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("scale", ctypes.c_float), ("flags", ctypes.c_uint32), ("state_scales", ctypes.c_void_p)]


class ChunkGrads(ctypes.Structure):
    _fields_ = [("dout", ctypes.c_void_p), ("dhT", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p), ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p), ("dh0", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libgdnqat.so (building it in-tree if it is missing and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB_PATH) or (build_if_missing and not _build.up_to_date()):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {_build.LIB_PATH}")
            _build.build()
        lib = ctypes.CDLL(_build.LIB_PATH)
        P, I32, U32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float
        for fn in ("gdn_chunk_fwd_workspace_size", "kda_chunk_fwd_workspace_size",
                   "gdn_prefill_decode_workspace_size", "kda_prefill_decode_workspace_size"):
            getattr(lib, fn).restype = ctypes.c_size_t
            getattr(lib, fn).argtypes = [ctypes.POINTER(ChunkArgs)]
        for fn in ("gdn_chunk_fwd", "kda_chunk_fwd"):
            getattr(lib, fn).restype = ctypes.c_int
            getattr(lib, fn).argtypes = [ctypes.POINTER(ChunkArgs), P, ctypes.c_size_t, P]
        for fn in ("gdn_chunk_bwd_workspace_size", "kda_chunk_bwd_workspace_size"):
            getattr(lib, fn).restype = ctypes.c_size_t
            getattr(lib, fn).argtypes = [ctypes.POINTER(ChunkArgs)]
        for fn in ("gdn_chunk_bwd", "kda_chunk_bwd"):
            getattr(lib, fn).restype = ctypes.c_int
            getattr(lib, fn).argtypes = [ctypes.POINTER(ChunkArgs), ctypes.POINTER(ChunkGrads), P, ctypes.c_size_t, P]
        for fn in ("gdn_prefill_decode_fwd", "kda_prefill_decode_fwd"):
            getattr(lib, fn).restype = ctypes.c_int
            getattr(lib, fn).argtypes = [ctypes.POINTER(ChunkArgs), P, P, ctypes.c_size_t, P]
        lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.gdn_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(ChunkArgs), P]
        lib.gdn_decode_step.restype = ctypes.c_int
        lib.gdn_decode_step.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, I32, F, U32, P]
        lib.fp8_tile_qdq.restype = ctypes.c_int
        lib.fp8_tile_qdq.argtypes = [P, P, P, ctypes.c_int64, I32, I32, I32, P]
        lib.int8_block_qdq.restype = ctypes.c_int
        lib.int8_block_qdq.argtypes = [P, P, P, ctypes.c_int64, I32, I32, P]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_check_device_status.restype = ctypes.c_int
        lib.gdn_check_device_status.argtypes = [P, P]
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _check(fn, st):
    if st != GDN_OK:
        raise GdnError(fn, st)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _state_flags(state_qdq, codec):
    """GDN_FLAG_STATE_QDQ (and GDN_FLAG_STATE_INT8 for codec "int8")."""
    if codec not in ("e4m3", "int8"):
        raise ValueError(f"unknown state codec {codec!r}")
    if not state_qdq:
        return 0
    return GDN_FLAG_STATE_QDQ | (GDN_FLAG_STATE_INT8 if codec == "int8" else 0)


def _dev(t, dtype, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def workspace_bytes(args: ChunkArgs, kda: bool = False) -> int:
    fn = "kda_chunk_fwd_workspace_size" if kda else "gdn_chunk_fwd_workspace_size"
    return int(getattr(load(), fn)(ctypes.byref(args)))


def chunk_workspace_bytes(q_shape, v_shape, cu_seqlens=None, *, state_qdq=False, w_qdq=False, kda=False):
    """gdn_chunk_fwd_workspace_size (kda: kda_chunk_fwd_workspace_size) for q [B,T,Hqk,dk],
    v [B,T,Hv,dv] (shapes only): the workspace of the fastest path. The size depends on shapes
    and flags only, so the query passes distinct placeholder device addresses."""
    B, T, Hqk, dk = q_shape
    Hv, dv = v_shape[2], v_shape[3]
    cu_host, N = None, B
    if cu_seqlens is not None:
        cu_host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        N = cu_host.numel() - 1
    fake = [ctypes.c_void_p((1 << 44) + (i << 38)) for i in range(10)]
    flags = (GDN_FLAG_STATE_QDQ if state_qdq else 0) | (GDN_FLAG_W_QDQ if w_qdq else 0)
    a = ChunkArgs(fake[0], fake[1], fake[2], fake[3], fake[4], None, fake[6] if cu_host is not None else None,
                  _ptr(cu_host), fake[8], fake[9], B, T, N, Hqk, Hv, dk, dv, 1.0, flags)
    return workspace_bytes(a, kda)


def _chunk_args(q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT, output_final_state, codec="e4m3",
                state_scales=None):
    q = _dev(q, torch.bfloat16, "q")
    k = _dev(k, torch.bfloat16, "k")
    v = _dev(v, torch.bfloat16, "v")
    g = _dev(g, torch.float32, "g")
    beta = _dev(beta, torch.float32, "beta")
    h0 = _dev(h0, torch.float32, "h0")
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    dev = q.device
    cu_dev = cu_host = None
    if cu_seqlens is not None:
        cu_host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        cu_dev = cu_seqlens.to(dev, torch.int32).contiguous() if cu_seqlens.is_cuda else cu_host.to(dev)
        N = cu_host.numel() - 1
    else:
        N = B
    if o is None:
        o = torch.empty((B, T, Hv, dv), dtype=torch.float32, device=dev)
    if hT is None and output_final_state:
        hT = torch.empty((N, Hv, dk, dv), dtype=torch.float32, device=dev)
    flags = _state_flags(state_qdq, codec) | (GDN_FLAG_W_QDQ if w_qdq else 0)
    # the host copy of cu_seqlens must outlive the call: it is returned with the args
    state_scales = _dev(state_scales, torch.float32, "state_scales")
    a = ChunkArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_dev), _ptr(cu_host),
                  _ptr(o), _ptr(hT), B, T, N, Hqk, Hv, dk, dv, float(scale), flags, _ptr(state_scales))
    return a, (o, hT), (cu_host, cu_dev)


def _chunk(fn_name, q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT, output_final_state,
           workspace, stream, codec="e4m3", state_scales=None):
    lib = load()
    a, (o, hT), _keep = _chunk_args(q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT,
                                    output_final_state, codec, state_scales)
    dev = o.device
    need = workspace_bytes(a, fn_name == "kda_chunk_fwd")
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = getattr(lib, fn_name)(ctypes.byref(a), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(fn_name, st)
    return o, hT


def gdn_chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, *, state_qdq=False, w_qdq=False, scale=1.0,
                  o=None, hT=None, output_final_state=True, workspace=None, stream=None, codec="e4m3",
                  state_scales=None):
    """Chunked GDN forward. q, k [B,T,Hqk,dk] bf16; v [B,T,Hv,dv] bf16; g, beta [B,T,Hv] fp32;
    h0 [N,Hv,dk,dv] fp32 or None; cu_seqlens int32 [N+1] (CPU or CUDA) or None; codec: the state
    QDQ format, "e4m3" (tiles) or "int8" (blocks of 32 value columns per key row); state_scales:
    an fp32 CUDA tensor that receives the final state's QDQ scales ([N,Hv,dv/64], INT8
    [N,Hv,dk,dv/32]; 0 where not QDQ'd) or None.
    Returns (o [B,T,Hv,dv] fp32, hT [N,Hv,dk,dv] fp32 or None)."""
    return _chunk("gdn_chunk_fwd", q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT,
                  output_final_state, workspace, stream, codec, state_scales)


def kda_chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, *, state_qdq=False, w_qdq=False, scale=1.0,
                  o=None, hT=None, output_final_state=True, workspace=None, stream=None, codec="e4m3",
                  state_scales=None):
    """KDA chunked forward: as gdn_chunk_fwd with g [B,T,Hv,dk] (one log-decay per key channel)."""
    return _chunk("kda_chunk_fwd", q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT,
                  output_final_state, workspace, stream, codec, state_scales)


def prefill_decode_workspace_bytes(q_shape, v_shape, cu_seqlens=None, *, state_qdq=False, w_qdq=False, kda=False):
    """gdn_prefill_decode_workspace_size (kda: kda_prefill_decode_workspace_size) for these shapes."""
    B, T, Hqk, dk = q_shape
    Hv, dv = v_shape[2], v_shape[3]
    cu_host, N = None, B
    if cu_seqlens is not None:
        cu_host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        N = cu_host.numel() - 1
    fake = [ctypes.c_void_p((1 << 44) + (i << 38)) for i in range(10)]
    flags = (GDN_FLAG_STATE_QDQ if state_qdq else 0) | (GDN_FLAG_W_QDQ if w_qdq else 0)
    a = ChunkArgs(fake[0], fake[1], fake[2], fake[3], fake[4], None, fake[6] if cu_host is not None else None,
                  _ptr(cu_host), fake[8], fake[9], B, T, N, Hqk, Hv, dk, dv, 1.0, flags)
    fn = "kda_prefill_decode_workspace_size" if kda else "gdn_prefill_decode_workspace_size"
    return int(getattr(load(), fn)(ctypes.byref(a)))


def _prefill_decode(fn_name, q, k, v, g, beta, h0, cu_seqlens, prefill_lengths, state_qdq, w_qdq, scale, o, hT,
                    workspace, stream, codec="e4m3", state_scales=None):
    lib = load()
    a, (o, hT), _keep = _chunk_args(q, k, v, g, beta, h0, cu_seqlens, state_qdq, w_qdq, scale, o, hT, True, codec,
                                    state_scales)
    pl = torch.as_tensor(prefill_lengths, dtype=torch.int32).to("cpu").contiguous().reshape(-1)
    if pl.numel() != a.N:
        raise ValueError(f"prefill_lengths: {pl.numel()} entries for {a.N} sequences")
    dev = o.device
    size_fn = "kda_prefill_decode_workspace_size" if fn_name == "kda_prefill_decode_fwd" else \
        "gdn_prefill_decode_workspace_size"
    need = int(getattr(lib, size_fn)(ctypes.byref(a)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = getattr(lib, fn_name)(ctypes.byref(a), _ptr(pl), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(fn_name, st)
    return o, hT


def gdn_prefill_decode_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, prefill_lengths=None, *, state_qdq=False,
                           w_qdq=False, scale=1.0, o=None, hT=None, workspace=None, stream=None, codec="e4m3",
                           state_scales=None):
    """Prefill -> decode handoff: per sequence the first prefill_lengths[n] tokens chunked with no
    state QDQ, then (state_qdq) a QDQ at the handoff and one decode step with state QDQ per
    remaining token. Same tensors as gdn_chunk_fwd; prefill_lengths: N ints (host).
    Returns (o, hT)."""
    return _prefill_decode("gdn_prefill_decode_fwd", q, k, v, g, beta, h0, cu_seqlens, prefill_lengths, state_qdq,
                           w_qdq, scale, o, hT, workspace, stream, codec, state_scales)


def kda_prefill_decode_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, prefill_lengths=None, *, state_qdq=False,
                           w_qdq=False, scale=1.0, o=None, hT=None, workspace=None, stream=None, codec="e4m3",
                           state_scales=None):
    """The handoff schedule for KDA (g [B,T,Hv,dk])."""
    return _prefill_decode("kda_prefill_decode_fwd", q, k, v, g, beta, h0, cu_seqlens, prefill_lengths, state_qdq,
                           w_qdq, scale, o, hT, workspace, stream, codec, state_scales)


def _chunk_bwd(fn_name, q, k, v, g, beta, h0, cu_seqlens, dout, dhT, state_qdq, scale, codec, want_dh0, workspace,
               stream):
    lib = load()
    dev = q.device
    # the forward's arguments (o and hT are not read by the backward)
    a, _, _keep = _chunk_args(q, k, v, g, beta, h0, cu_seqlens, state_qdq, False, scale,
                              torch.empty(0, device=dev), None, False, codec)
    a.o = None
    dout = _dev(dout, torch.float32, "dout")
    dhT = _dev(dhT, torch.float32, "dhT")
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
    dg = torch.empty(g.shape, dtype=torch.float32, device=dev)
    dbeta = torch.empty(beta.shape, dtype=torch.float32, device=dev)
    dh0 = torch.empty((a.N, a.Hv, a.dk, a.dv), dtype=torch.float32, device=dev) if want_dh0 else None
    gr = ChunkGrads(_ptr(dout), _ptr(dhT), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0))
    size_fn = fn_name + "_workspace_size"
    need = int(getattr(lib, size_fn)(ctypes.byref(a)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = getattr(lib, fn_name)(ctypes.byref(a), ctypes.byref(gr), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(fn_name, st)
    return dq, dk, dv, dg, dbeta, dh0


def gdn_chunk_bwd(q, k, v, g, beta, h0=None, cu_seqlens=None, dout=None, dhT=None, *, state_qdq=False, scale=1.0,
                  codec="e4m3", want_dh0=True, workspace=None, stream=None):
    """Gradients of <o, dout> + <hT, dhT> for the forward with straight-through state QDQ (no W QDQ).
    Inputs as gdn_chunk_fwd; dout [B,T,Hv,dv] fp32; dhT [N,Hv,dk,dv] fp32 or None.
    Returns (dq, dk, dv, dg, dbeta, dh0) fp32 (dh0 None unless want_dh0)."""
    return _chunk_bwd("gdn_chunk_bwd", q, k, v, g, beta, h0, cu_seqlens, dout, dhT, state_qdq, scale, codec, want_dh0,
                      workspace, stream)


def kda_chunk_bwd(q, k, v, g, beta, h0=None, cu_seqlens=None, dout=None, dhT=None, *, state_qdq=False, scale=1.0,
                  codec="e4m3", want_dh0=True, workspace=None, stream=None):
    """The KDA backward (g and dg [B,T,Hv,dk])."""
    return _chunk_bwd("kda_chunk_bwd", q, k, v, g, beta, h0, cu_seqlens, dout, dhT, state_qdq, scale, codec, want_dh0,
                      workspace, stream)


def chunk_bwd_workspace_bytes(q_shape, v_shape, cu_seqlens=None, *, kda=False):
    """gdn_chunk_bwd_workspace_size (kda: kda_chunk_bwd_workspace_size) for these shapes."""
    B, T, Hqk, dk = q_shape
    Hv, dv = v_shape[2], v_shape[3]
    cu_host, N = None, B
    if cu_seqlens is not None:
        cu_host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        N = cu_host.numel() - 1
    fake = [ctypes.c_void_p((1 << 44) + (i << 38)) for i in range(10)]
    a = ChunkArgs(fake[0], fake[1], fake[2], fake[3], fake[4], None, fake[6] if cu_host is not None else None,
                  _ptr(cu_host), None, None, B, T, N, Hqk, Hv, dk, dv, 1.0, GDN_FLAG_STATE_QDQ)
    fn = "kda_chunk_bwd_workspace_size" if kda else "gdn_chunk_bwd_workspace_size"
    return int(getattr(load(), fn)(ctypes.byref(a)))


def gdn_decode_step(q, k, v, g, beta, state, *, state_qdq=True, kda=False, scale=1.0, o=None, stream=None,
                    codec="e4m3"):
    """One decode token per sequence; `state` [N,Hv,dk,dv] fp32 is updated in place.
    q, k [N,Hqk,dk] bf16; v [N,Hv,dv] bf16; g [N,Hv] (kda: [N,Hv,dk]) fp32; beta [N,Hv] fp32.
    Returns o [N,Hv,dv] fp32."""
    lib = load()
    q = _dev(q, torch.bfloat16, "q")
    k = _dev(k, torch.bfloat16, "k")
    v = _dev(v, torch.bfloat16, "v")
    g = _dev(g, torch.float32, "g")
    beta = _dev(beta, torch.float32, "beta")
    state = _dev(state, torch.float32, "state")
    N, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    if o is None:
        o = torch.empty((N, Hv, dv), dtype=torch.float32, device=q.device)
    flags = _state_flags(state_qdq, codec) | (GDN_FLAG_KDA if kda else 0)
    st = lib.gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(o), N, Hqk, Hv,
                             dk, dv, float(scale), flags, _stream(stream, q.device))
    _check("gdn_decode_step", st)
    return o


def fp8_tile_qdq(x, tile_cols, *, y=None, scales=True, stream=None):
    """Dynamic per-tile E4M3 QDQ of x [lead, rows, cols] fp32 (a tile = all rows x tile_cols
    columns). Returns (y, scales [lead, ceil(cols/tile_cols)] or None). y may be x."""
    lib = load()
    x = _dev(x, torch.float32, "x")
    if x.dim() == 2:
        x = x.unsqueeze(0)
    lead, rows, cols = x.shape
    if y is None:
        y = torch.empty_like(x)
    sc = None
    if scales:
        sc = torch.empty((lead, (cols + tile_cols - 1) // tile_cols), dtype=torch.float32, device=x.device)
    st = lib.fp8_tile_qdq(_ptr(x), _ptr(y), _ptr(sc), lead, rows, cols, int(tile_cols), _stream(stream, x.device))
    _check("fp8_tile_qdq", st)
    return y, sc


def int8_block_qdq(x, block_cols=32, *, y=None, scales=True, stream=None):
    """INT8 block QDQ of x (fp32, last dimension = columns; leading dimensions are rows): one
    scale per block_cols consecutive columns of a row. Returns (y, scales [rows, ceil(cols /
    block_cols)] or None). y may be x."""
    lib = load()
    x = _dev(x, torch.float32, "x")
    cols = x.shape[-1] if x.dim() else 1
    rows = x.numel() // cols if cols else 0
    if y is None:
        y = torch.empty_like(x)
    sc = None
    if scales:
        sc = torch.empty((rows, (cols + block_cols - 1) // block_cols), dtype=torch.float32, device=x.device)
    st = lib.int8_block_qdq(_ptr(x), _ptr(y), _ptr(sc), rows, cols, int(block_cols), _stream(stream, x.device))
    _check("int8_block_qdq", st)
    return y, sc


def gdn_check_device_status(workspace, stream=None):
    """Raise GdnError if a kernel that used `workspace` gave up a bounded wait. workspace None:
    the library array behind gdn_chunk_fwd_noalloc on the current device."""
    dev = workspace.device if workspace is not None else torch.device("cuda", torch.cuda.current_device())
    st = load().gdn_check_device_status(_ptr(workspace), _stream(stream, dev))
    _check("gdn_check_device_status", st)
