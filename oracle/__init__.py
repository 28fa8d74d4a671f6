"""fp64 CPU oracle for the chunked gated-delta-rule forward with FP8 E4M3 state QDQ.

TEST INFRASTRUCTURE ONLY: the plain, slow, independent reference that the CUDA library
is checked against. Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library
(``fp8_state_qat_gb300``) and never consumes anything that library produced.

The arithmetic lives in ``gdn_oracle.cpp`` (C++17, fp64); this module only builds it with
g++ and marshals numpy arrays through ctypes. Sources for every step are cited in the C++
file: "GDN state/W QAT foundation" (state and W QDQ contract), "Torch GDN/KDA decode QAT
with INT8 recurrent state" (decode order), "Add KDA prefill numerical emulation for QAT"
(per-key-channel retention), "Add experimental GDN/KDA decode and replay QAT" (per-token
state writes). Every prefill / decode function takes ``codec``: the state QDQ format, "e4m3"
(tiles of all dk rows x 64 value columns) or "int8" (blocks of one key row x 32 value columns).

Pins: every function here is checked in tests/test_oracle_*.py against closed forms,
invariants, hand-worked examples and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libgdn_oracle.so`` (g++, fp64, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_e4m3_rne.restype = D
            lib.oracle_e4m3_rne.argtypes = [D]
            lib.oracle_tile_qdq_f32.restype = I
            lib.oracle_tile_qdq_f32.argtypes = [P, P, P, ctypes.c_int64, I, I, I]
            lib.oracle_tile_qdq_f64.restype = I
            lib.oracle_tile_qdq_f64.argtypes = [P, P, ctypes.c_int64, I, I, I]
            lib.oracle_gdn_recurrent.restype = I
            lib.oracle_gdn_recurrent.argtypes = [P] * 7 + [I] * 10 + [D, P, I, P, P]
            lib.oracle_gdn_chunked.restype = I
            lib.oracle_gdn_chunked.argtypes = [P] * 7 + [I] * 11 + [D, P, I, P, P]
            lib.oracle_gdn_decode.restype = I
            lib.oracle_gdn_decode.argtypes = [P] * 5 + [I] * 8 + [D, P, I, P, P]
            lib.oracle_int8_block_qdq_f32.restype = I
            lib.oracle_int8_block_qdq_f32.argtypes = [P, P, P, ctypes.c_int64, I, I]
            lib.oracle_int8_block_qdq_f64.restype = I
            lib.oracle_int8_block_qdq_f64.argtypes = [P, P, ctypes.c_int64, I, I]
            lib.oracle_gdn_prefill_decode.restype = I
            lib.oracle_gdn_prefill_decode.argtypes = [P] * 8 + [I] * 10 + [D, P, I, P, P]
            _lib = lib
    return _lib


def _f32(x):
    """torch tensor or array -> C-contiguous float32 numpy array (bf16 widens exactly)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float32).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def e4m3_rne(y: float) -> float:
    """E4M3 (fn) round-to-nearest-even with saturation to +-448, in fp64."""
    return _load().oracle_e4m3_rne(float(y))


def tile_qdq_f32(x, tile_cols: int):
    """fp32 tile QDQ of x [lead, rows, cols]. Returns (y fp32, scales fp32 [lead, ntiles])."""
    x = _f32(x)
    if x.ndim == 2:
        x = x[None]
    lead, rows, cols = x.shape
    ntiles = (cols + tile_cols - 1) // tile_cols if cols else 0
    y = np.empty_like(x)
    sc = np.empty((lead, ntiles), np.float32)
    rc = _load().oracle_tile_qdq_f32(_ptr(x), _ptr(y), _ptr(sc), lead, rows, cols, tile_cols)
    if rc:
        raise ValueError("oracle_tile_qdq_f32: bad arguments")
    return y, sc


def tile_qdq_f64(x, tile_cols: int):
    """The same tile QDQ in fp64. Returns (y fp64, scales fp64)."""
    y = np.array(x, dtype=np.float64, copy=True, order="C")
    if y.ndim == 2:
        y = y[None]
    lead, rows, cols = y.shape
    ntiles = (cols + tile_cols - 1) // tile_cols if cols else 0
    sc = np.empty((lead, ntiles), np.float64)
    rc = _load().oracle_tile_qdq_f64(_ptr(y), _ptr(sc), lead, rows, cols, tile_cols)
    if rc:
        raise ValueError("oracle_tile_qdq_f64: bad arguments")
    return y, sc


def _codec(state_qdq, codec):
    """The oracle's state-QDQ selector: 0 off, 1 E4M3 tiles, 2 INT8 blocks of 32 value columns."""
    if not state_qdq:
        return 0
    if codec not in ("e4m3", "int8"):
        raise ValueError(f"unknown state codec {codec!r}")
    return 2 if codec == "int8" else 1


def int8_block_qdq_f32(x, block_cols: int = 32):
    """INT8 block QDQ of x [rows, cols] (any leading shape is flattened into rows) in fp32.
    Returns (y fp32, scales fp32 [rows, ceil(cols / block_cols)])."""
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    cols = xa.shape[-1] if xa.ndim else 1
    rows = xa.size // cols if cols else 0
    y = np.empty_like(xa)
    nb = (cols + block_cols - 1) // block_cols if cols else 0
    sc = np.empty((rows, nb), np.float32)
    rc = _load().oracle_int8_block_qdq_f32(_ptr(xa), _ptr(y), _ptr(sc), rows, cols, block_cols)
    if rc:
        raise ValueError("oracle_int8_block_qdq_f32: bad arguments")
    return y, sc


def int8_block_qdq_f64(x, block_cols: int = 32):
    """The INT8 block codec in fp64. Returns (y fp64, scales fp64)."""
    y = np.array(x, dtype=np.float64, copy=True, order="C")
    cols = y.shape[-1] if y.ndim else 1
    rows = y.size // cols if cols else 0
    nb = (cols + block_cols - 1) // block_cols if cols else 0
    sc = np.empty((rows, nb), np.float64)
    rc = _load().oracle_int8_block_qdq_f64(_ptr(y), _ptr(sc), rows, cols, block_cols)
    if rc:
        raise ValueError("oracle_int8_block_qdq_f64: bad arguments")
    return y, sc


def _prefill_args(q, k, v, g, beta, h0, cu_seqlens, kda):
    q, k, v, g, beta = (_f32(t) for t in (q, k, v, g, beta))
    h0 = _f64(h0)
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    cu = None
    if cu_seqlens is not None:
        c = cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens
        cu = np.ascontiguousarray(np.asarray(c, dtype=np.int32))
        N = cu.shape[0] - 1
    else:
        N = B
    if kda:
        assert g.shape == (B, T, Hv, dk), g.shape
    else:
        assert g.shape == (B, T, Hv), g.shape
    return q, k, v, g, beta, h0, cu, B, T, N, Hqk, Hv, dk, dv


def _mask(unit_mask, N, Hv):
    if unit_mask is None:
        return None
    return np.ascontiguousarray(np.asarray(unit_mask, dtype=np.uint8).reshape(N * Hv))


def gdn_recurrent(q, k, v, g, beta, h0=None, cu_seqlens=None, *, kda=False, state_qdq=False,
                  qdq_period=64, scale=1.0, unit_mask=None, threads=None, codec="e4m3"):
    """O1: token-by-token fp64 recurrence. Returns (o [B,T,Hv,dv], hT [N,Hv,dk,dv]) fp64."""
    q, k, v, g, beta, h0, cu, B, T, N, Hqk, Hv, dk, dv = _prefill_args(q, k, v, g, beta, h0, cu_seqlens, kda)
    o = np.zeros((B, T, Hv, dv), np.float64)
    hT = np.zeros((N, Hv, dk, dv), np.float64)
    m = _mask(unit_mask, N, Hv)
    rc = _load().oracle_gdn_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                                      B, T, N, Hqk, Hv, dk, dv, int(kda), _codec(state_qdq, codec), int(qdq_period),
                                      float(scale), _ptr(m), _threads(threads), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle_gdn_recurrent: bad arguments")
    return o, hT


def gdn_chunked(q, k, v, g, beta, h0=None, cu_seqlens=None, *, kda=False, chunk=64, state_qdq=False,
                w_qdq=False, scale=1.0, unit_mask=None, threads=None, codec="e4m3"):
    """O2: chunked / WY fp64 form (needed for W QDQ). Returns (o, hT) fp64."""
    q, k, v, g, beta, h0, cu, B, T, N, Hqk, Hv, dk, dv = _prefill_args(q, k, v, g, beta, h0, cu_seqlens, kda)
    o = np.zeros((B, T, Hv, dv), np.float64)
    hT = np.zeros((N, Hv, dk, dv), np.float64)
    m = _mask(unit_mask, N, Hv)
    rc = _load().oracle_gdn_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                                    B, T, N, Hqk, Hv, dk, dv, int(kda), int(chunk), _codec(state_qdq, codec), int(w_qdq),
                                    float(scale), _ptr(m), _threads(threads), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle_gdn_chunked: bad arguments")
    return o, hT


def gdn_decode(q, k, v, g, beta, state, *, kda=False, state_qdq=True, scale=1.0, unit_mask=None,
               threads=None, codec="e4m3"):
    """Decode steps. q,k [steps,N,Hqk,dk]; v [steps,N,Hv,dv]; g [steps,N,Hv] (KDA [..,dk]);
    beta [steps,N,Hv]; state [N,Hv,dk,dv] (copied to fp64). Returns (o fp64, final state fp64)."""
    q, k, v, g, beta = (_f32(t) for t in (q, k, v, g, beta))
    steps, N, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    st = np.array(_f64(state), dtype=np.float64, copy=True, order="C")
    o = np.zeros((steps, N, Hv, dv), np.float64)
    m = _mask(unit_mask, N, Hv)
    rc = _load().oracle_gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), steps, N, Hqk, Hv, dk, dv,
                                   int(kda), _codec(state_qdq, codec), float(scale), _ptr(m), _threads(threads),
                                   _ptr(st), _ptr(o))
    if rc:
        raise ValueError("oracle_gdn_decode: bad arguments")
    return o, st


def gdn_prefill_decode(q, k, v, g, beta, h0=None, cu_seqlens=None, prefill_lengths=None, *, kda=False,
                       state_qdq=False, w_qdq=False, scale=1.0, unit_mask=None, threads=None, codec="e4m3"):
    """Prefill -> decode handoff: per sequence the first prefill_lengths[n] tokens chunked with no
    state QDQ, QDQ at the handoff when tokens remain, then one decode step (with state QDQ) per
    remaining token. Returns (o, hT) fp64."""
    q, k, v, g, beta, h0, cu, B, T, N, Hqk, Hv, dk, dv = _prefill_args(q, k, v, g, beta, h0, cu_seqlens, kda)
    pl = np.ascontiguousarray(np.asarray(prefill_lengths, dtype=np.int32).reshape(N))
    o = np.zeros((B, T, Hv, dv), np.float64)
    hT = np.zeros((N, Hv, dk, dv), np.float64)
    m = _mask(unit_mask, N, Hv)
    rc = _load().oracle_gdn_prefill_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                                           _ptr(pl), B, T, N, Hqk, Hv, dk, dv, int(kda), _codec(state_qdq, codec), int(w_qdq),
                                           float(scale), _ptr(m), _threads(threads), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle_gdn_prefill_decode: bad arguments")
    return o, hT
