"""The C ABI library (CPU-only checks): it builds, loads, exports every function that
include/gdnqat.h declares, and its host-side validation returns the documented status
before touching a device ("GDN state/W QAT foundation": errors are raised before any
kernel launches). No compute call is made here: the pointers are fake, so a call that passes
validation is made only where no GPU is present (it then stops at the device check)."""
import ctypes
import os
import re

import pytest
import torch

import fp8_state_qat_gb300 as lib
from fp8_state_qat_gb300 import gdnqat as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdnqat.h")


@pytest.fixture(scope="module")
def so():
    return lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def test_exports_every_declared_symbol(so):
    names = declared_functions()
    assert set(names) == set(B.EXPORTED), names
    for n in names:
        assert hasattr(so, n), n


def test_status_strings(so):
    for code in range(7):
        assert lib.status_string(code)
    assert lib.status_string(99) == "unknown status"


FAKE = 1 << 40   # distinct, 256-byte aligned fake device addresses; validation never dereferences them


def good_args(**over):
    a = dict(q=FAKE, k=FAKE + (1 << 32), v=FAKE + (2 << 32), g=FAKE + (3 << 32), beta=FAKE + (4 << 32), h0=None,
             cu_seqlens=None, cu_seqlens_host=None, o=FAKE + (5 << 32), hT=FAKE + (6 << 32),
             B=2, T=128, N=2, Hqk=2, Hv=4, dk=128, dv=128, scale=1.0, flags=3)
    a.update(over)
    return B.ChunkArgs(**a)


def call_chunk(so, args, ws=FAKE + (7 << 32), ws_bytes=1 << 20):
    return so.gdn_chunk_fwd(ctypes.byref(args), ctypes.c_void_p(ws), ws_bytes, None)


@pytest.mark.parametrize("over,want", [
    (dict(dk=96), B.GDN_ERR_UNSUPPORTED_SHAPE),
    (dict(dv=96), B.GDN_ERR_UNSUPPORTED_SHAPE),
    (dict(dv=512), B.GDN_ERR_UNSUPPORTED_SHAPE),
    (dict(Hv=3), B.GDN_ERR_INVALID_ARG),          # Hv % Hqk != 0
    (dict(N=3), B.GDN_ERR_INVALID_ARG),           # dense needs N == B
    (dict(q=None), B.GDN_ERR_INVALID_ARG),
    (dict(q=FAKE + 2), B.GDN_ERR_INVALID_ARG),    # misaligned
    (dict(flags=16), B.GDN_ERR_INVALID_ARG),      # unknown flag
    (dict(o=FAKE + (2 << 32) + 64), B.GDN_ERR_INVALID_ARG),   # o overlaps v
    (dict(h0=FAKE + (8 << 32), hT=FAKE + (8 << 32) + 256), B.GDN_ERR_INVALID_ARG),  # partial alias
])
def test_chunk_validation(so, over, want):
    assert call_chunk(so, good_args(**over)) == want


def test_varlen_validation(so):
    cu_bad = (ctypes.c_int32 * 4)(0, 50, 40, 128)   # non-monotone
    a = good_args(B=1, N=3, cu_seqlens=FAKE + (9 << 32), cu_seqlens_host=ctypes.addressof(cu_bad))
    assert call_chunk(so, a) == B.GDN_ERR_INVALID_ARG
    cu_end = (ctypes.c_int32 * 4)(0, 50, 60, 127)   # does not end at T
    a = good_args(B=1, N=3, cu_seqlens=FAKE + (9 << 32), cu_seqlens_host=ctypes.addressof(cu_end))
    assert call_chunk(so, a) == B.GDN_ERR_INVALID_ARG
    a = good_args(B=1, N=3, cu_seqlens=FAKE + (9 << 32), cu_seqlens_host=None)   # host copy required
    assert call_chunk(so, a) == B.GDN_ERR_INVALID_ARG


MIN_WS = 256   # GDN_CHUNK_MIN_WORKSPACE_BYTES


def test_workspace_checks(so):
    """Below the minimum (the status word) the call is refused before anything else; between
    the minimum and gdn_chunk_fwd_workspace_size() it is accepted (single-kernel path)."""
    a = good_args()
    assert call_chunk(so, a, ws_bytes=MIN_WS - 1) == B.GDN_ERR_WORKSPACE_TOO_SMALL
    assert call_chunk(so, a, ws=0) == B.GDN_ERR_WORKSPACE_TOO_SMALL
    # with enough workspace the next check is the device's (where there is none); with a GPU the
    # call would go on to use the fake addresses, so it is made only without one
    if not torch.cuda.is_available():
        assert call_chunk(so, a, ws_bytes=MIN_WS) == B.GDN_ERR_UNSUPPORTED_ARCH
    assert so.gdn_chunk_fwd_workspace_size(ctypes.byref(good_args(dk=96))) == 0


def test_workspace_size_covers_the_two_kernel_staging(so):
    """dk = 128: status word + per (chunk slot, v-head) W^T (16 KB with W QDQ, 32 KB without),
    T'' hi + lo (16 KB), P hi + lo (16 KB) and the gate vectors (1 KB), slots = B T / 64 + N.
    dk = 64: the minimum."""
    for flags, wt in ((B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_W_QDQ, 16), (B.GDN_FLAG_STATE_QDQ, 32)):
        a = good_args(flags=flags)
        items = (a.B * a.T // 64 + a.N) * a.Hv
        need = so.gdn_chunk_fwd_workspace_size(ctypes.byref(a))
        assert need >= MIN_WS + items * (wt + 16 + 16 + 1) * 1024
        assert need <= MIN_WS + items * (wt + 16 + 16 + 1) * 1024 + 5 * 1024
    assert so.gdn_chunk_fwd_workspace_size(ctypes.byref(good_args(dk=64))) == MIN_WS


def test_kda_workspace_size_covers_the_two_kernel_staging(so):
    """KDA, dk = 128: status word + per (chunk slot, v-head) W^T (16 / 32 KB), T'' (16 KB), P
    (16 KB), Q and K times their per-channel decays (32 KB each, bf16 hi + lo) and the decay
    vectors (1 KB). dk = 64: the minimum (CUDA-core path); invalid arguments: 0."""
    for flags, wt in ((B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_W_QDQ, 16), (B.GDN_FLAG_STATE_QDQ, 32)):
        a = good_args(flags=flags)
        items = (a.B * a.T // 64 + a.N) * a.Hv
        need = so.kda_chunk_fwd_workspace_size(ctypes.byref(a))
        per = (wt + 16 + 16 + 32 + 32 + 1) * 1024
        assert MIN_WS + items * per <= need <= MIN_WS + items * per + 8 * 1024
    assert so.kda_chunk_fwd_workspace_size(ctypes.byref(good_args(dk=64))) == MIN_WS
    assert so.kda_chunk_fwd_workspace_size(ctypes.byref(good_args(dk=96))) == 0
    # the binding's shape-only query agrees with the C call
    a = good_args(flags=B.GDN_FLAG_STATE_QDQ)
    q_shape, v_shape = (a.B, a.T, a.Hqk, a.dk), (a.B, a.T, a.Hv, a.dv)
    assert B.chunk_workspace_bytes(q_shape, v_shape, state_qdq=True, kda=True) == \
        so.kda_chunk_fwd_workspace_size(ctypes.byref(a))


def test_decode_and_qdq_validation(so):
    P = ctypes.c_void_p
    ptrs = [P(FAKE + (i << 32)) for i in range(7)]
    assert so.gdn_decode_step(*ptrs, 4, 2, 4, 96, 128, 1.0, 1, None) == B.GDN_ERR_UNSUPPORTED_SHAPE
    assert so.gdn_decode_step(*ptrs, 4, 3, 4, 128, 128, 1.0, 1, None) == B.GDN_ERR_INVALID_ARG
    assert so.gdn_decode_step(*ptrs, 4, 2, 4, 128, 128, 1.0, 16, None) == B.GDN_ERR_INVALID_ARG
    assert so.fp8_tile_qdq(P(FAKE), P(FAKE), None, 2, 8, 64, 0, None) == B.GDN_ERR_INVALID_ARG
    assert so.fp8_tile_qdq(P(FAKE), P(FAKE + 4), None, 2, 8, 64, 64, None) == B.GDN_ERR_INVALID_ARG  # overlap


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_args_without_device_report_arch(so):
    assert call_chunk(so, good_args()) == B.GDN_ERR_UNSUPPORTED_ARCH
    P = ctypes.c_void_p
    ptrs = [P(FAKE + (i << 32)) for i in range(7)]
    assert so.gdn_decode_step(*ptrs, 4, 2, 4, 128, 128, 1.0, 1, None) == B.GDN_ERR_UNSUPPORTED_ARCH
    assert so.fp8_tile_qdq(P(FAKE), P(FAKE), None, 2, 8, 64, 64, None) == B.GDN_ERR_UNSUPPORTED_ARCH


def call_handoff(so, args, plens, ws=FAKE + (7 << 32), ws_bytes=1 << 30, kda=False):
    fn = so.kda_prefill_decode_fwd if kda else so.gdn_prefill_decode_fwd
    arr = None if plens is None else (ctypes.c_int32 * len(plens))(*plens)
    return fn(ctypes.byref(args), None if arr is None else ctypes.cast(arr, ctypes.c_void_p), ctypes.c_void_p(ws),
              ws_bytes, None)


def test_handoff_workspace_size(so):
    """The prefill's workspace (the two-kernel staging for dk = 128, the minimum otherwise),
    rounded up to 256 bytes, plus the device copy of the N prefill lengths."""
    for kda in (False, True):
        for over in (dict(), dict(dk=64)):
            a = good_args(**over)
            chunk = (so.kda_chunk_fwd_workspace_size if kda else so.gdn_chunk_fwd_workspace_size)(ctypes.byref(a))
            size = (so.kda_prefill_decode_workspace_size if kda else so.gdn_prefill_decode_workspace_size)
            assert size(ctypes.byref(a)) == (chunk + 255) // 256 * 256 + 4 * a.N
    assert so.gdn_prefill_decode_workspace_size(ctypes.byref(good_args(dk=96))) == 0
    a = good_args()
    assert B.prefill_decode_workspace_bytes((a.B, a.T, a.Hqk, a.dk), (a.B, a.T, a.Hv, a.dv), state_qdq=True,
                                            w_qdq=True) == so.gdn_prefill_decode_workspace_size(ctypes.byref(a))


def test_handoff_validation(so):
    """Prefill lengths outside [0, L_n], a missing hT or length array, and a workspace below the
    size query are refused before any device work (the next check is the device's: none here)."""
    for kda in (False, True):
        a = good_args()
        need = (so.kda_prefill_decode_workspace_size if kda else so.gdn_prefill_decode_workspace_size)(ctypes.byref(a))
        assert call_handoff(so, a, [129, 0], kda=kda) == B.GDN_ERR_INVALID_ARG
        assert call_handoff(so, a, [-1, 0], kda=kda) == B.GDN_ERR_INVALID_ARG
        assert call_handoff(so, a, None, kda=kda) == B.GDN_ERR_INVALID_ARG
        assert call_handoff(so, good_args(hT=None), [64, 64], kda=kda) == B.GDN_ERR_INVALID_ARG
        assert call_handoff(so, a, [64, 128], ws_bytes=need - 1, kda=kda) == B.GDN_ERR_WORKSPACE_TOO_SMALL
        if not torch.cuda.is_available():
            assert call_handoff(so, a, [64, 128], ws_bytes=need, kda=kda) == B.GDN_ERR_UNSUPPORTED_ARCH
    cu = (ctypes.c_int32 * 4)(0, 50, 60, 128)
    a = good_args(B=1, N=3, cu_seqlens=FAKE + (9 << 32), cu_seqlens_host=ctypes.addressof(cu))
    assert call_handoff(so, a, [50, 11, 0]) == B.GDN_ERR_INVALID_ARG   # 11 > L_1 = 10
    if not torch.cuda.is_available():
        assert call_handoff(so, a, [50, 10, 0]) == B.GDN_ERR_UNSUPPORTED_ARCH


def test_int8_codec_flags_and_standalone_validation(so):
    """GDN_FLAG_STATE_INT8 is accepted by the chunk, handoff and decode calls (the next check is
    the device's); the standalone INT8 op validates like the E4M3 one."""
    P = ctypes.c_void_p
    flags = B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_W_QDQ | B.GDN_FLAG_STATE_INT8
    want = B.GDN_ERR_UNSUPPORTED_ARCH if not torch.cuda.is_available() else None
    if want is not None:
        assert call_chunk(so, good_args(flags=flags)) == want
        ptrs = [P(FAKE + (i << 32)) for i in range(7)]
        assert so.gdn_decode_step(*ptrs, 4, 2, 4, 128, 128, 1.0, B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_STATE_INT8,
                                  None) == want
    assert so.int8_block_qdq(P(FAKE), P(FAKE), None, 2, 64, 0, None) == B.GDN_ERR_INVALID_ARG
    assert so.int8_block_qdq(P(FAKE), P(FAKE + 4), None, 2, 64, 32, None) == B.GDN_ERR_INVALID_ARG   # overlap
    assert so.int8_block_qdq(P(FAKE), P(FAKE), None, -1, 64, 32, None) == B.GDN_ERR_INVALID_ARG


def test_state_scales_validation(so):
    """The optional final-state scales need the state quantizer, 4-byte alignment and no overlap
    with o, h0 or hT."""
    assert call_chunk(so, good_args(flags=B.GDN_FLAG_W_QDQ, state_scales=FAKE + (10 << 32))) == B.GDN_ERR_INVALID_ARG
    assert call_chunk(so, good_args(state_scales=FAKE + (10 << 32) + 2)) == B.GDN_ERR_INVALID_ARG
    assert call_chunk(so, good_args(state_scales=FAKE + (5 << 32) + 64)) == B.GDN_ERR_INVALID_ARG   # inside o
    if not torch.cuda.is_available():
        assert call_chunk(so, good_args(state_scales=FAKE + (10 << 32))) == B.GDN_ERR_UNSUPPORTED_ARCH


def test_backward_validation(so):
    """The backward refuses W QDQ (its straight-through gradient belongs to the chunked form) and
    missing gradient buffers; its workspace covers the chunk-entry states and the per-CTA
    sub-chunk checkpoints of a 64-column slab (at most one CTA per SM)."""
    P = ctypes.c_void_p
    a = good_args(flags=B.GDN_FLAG_STATE_QDQ, o=None)
    need = so.gdn_chunk_bwd_workspace_size(ctypes.byref(a))
    slots = (a.B * a.T) // 64 + a.N
    state = a.dk * a.dv * 4
    slabs = a.dv // 64
    assert need >= 256 + slots * a.Hv * state + min(a.N * a.Hv * slabs, 152) * 16 * a.dk * 64 * 4
    assert so.gdn_chunk_bwd_workspace_size(ctypes.byref(good_args(flags=3))) == 0        # W QDQ
    # KDA adds a per-key-channel dg partial for every slab and (token, v-head)
    assert so.kda_chunk_bwd_workspace_size(ctypes.byref(a)) >= need + slabs * a.B * a.T * a.Hv * (a.dk - a.dk // 32) * 4
    g = B.ChunkGrads(*[P(FAKE + ((11 + i) << 32)) for i in range(8)])
    fn = so.gdn_chunk_bwd
    assert fn(ctypes.byref(good_args(flags=3, o=None)), ctypes.byref(g), P(FAKE + (7 << 32)), need,
              None) == B.GDN_ERR_INVALID_ARG
    g_missing = B.ChunkGrads(*[P(FAKE + ((11 + i) << 32)) for i in range(2)], None)
    assert fn(ctypes.byref(a), ctypes.byref(g_missing), P(FAKE + (7 << 32)), need, None) == B.GDN_ERR_INVALID_ARG
    assert fn(ctypes.byref(a), ctypes.byref(g), P(FAKE + (7 << 32)), need - 1, None) == B.GDN_ERR_WORKSPACE_TOO_SMALL
    # KDA stages g in 16-byte copies: a 4-byte aligned g is refused
    a_g4 = good_args(flags=B.GDN_FLAG_STATE_QDQ, o=None, g=FAKE + (3 << 32) + 4)
    kneed = so.kda_chunk_bwd_workspace_size(ctypes.byref(good_args(flags=B.GDN_FLAG_STATE_QDQ, o=None)))
    assert so.kda_chunk_bwd(ctypes.byref(a_g4), ctypes.byref(g), P(FAKE + (7 << 32)), kneed,
                            None) == B.GDN_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert fn(ctypes.byref(a), ctypes.byref(g), P(FAKE + (7 << 32)), need, None) == B.GDN_ERR_UNSUPPORTED_ARCH


def test_testing_library_builds_and_exports():
    """The test-only library (layout self-test, the chunk kernels with zero-poll waits) builds and
    exports its two entry points; the product library exports neither."""
    import native
    t = native.load()
    for name in ("gdnqat_internal_tc_selftest", "gdnqat_testing_split_fwd"):
        assert hasattr(t, name), name
        assert not hasattr(lib.load(), name), name


def test_check_device_status_null_reads_noalloc_array(so):
    """gdn_check_device_status(NULL) addresses the array behind gdn_chunk_fwd_noalloc; without a
    device it reports a CUDA error instead of reading anything."""
    if not torch.cuda.is_available():
        assert so.gdn_check_device_status(None, None) in (B.GDN_ERR_CUDA, B.GDN_ERR_UNSUPPORTED_ARCH)
