"""gdn_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate device memory
(for example code inside an allocator's own hooks, or a process whose device memory all
belongs to a framework pool). It takes its workspace from a small array inside the library
instead of a caller-provided buffer.

Checked through the C ABI on two calls in a row (the array keeps the previous call's
contents): bit for bit against gdn_chunk_fwd given the same 256-byte minimum workspace (both
run the same deterministic single-kernel path), against the fp64 oracle within the QDQ
tolerance, and the array's status word read back through gdn_check_device_status(NULL).
This file is collected last on purpose, so that a stop-at-first-failure run has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import gdnqat as B
from fp8_state_qat_gb300 import workloads
from helpers import TOL_QDQ, rel

pytestmark = pytest.mark.gpu


def _args(c, x, o, hT, flags):
    s = x.shape
    return B.ChunkArgs(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["g"].data_ptr(),
                       c["beta"].data_ptr(), c["h0"].data_ptr(), None, None, o.data_ptr(), hT.data_ptr(),
                       s["B"], s["T"], s["N"], s["Hqk"], s["Hv"], s["dk"], s["dv"], 1.0, flags)


def test_noalloc_matches_workspace_entry_point(gdn, oracle_mod):
    lib = gdn.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    flags = B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_W_QDQ
    for call, seed in enumerate((71, 72)):           # two calls in a row, different inputs
        x = workloads.prefill(2, 200, 2, 4, 128, 128, seed=seed, h0_std=0.1)
        c = {k: getattr(x, k).cuda() for k in ("q", "k", "v", "g", "beta", "h0")}
        s = x.shape
        o_ref = torch.empty((s["B"], s["T"], s["Hv"], s["dv"]), device="cuda")
        h_ref = torch.empty((s["N"], s["Hv"], s["dk"], s["dv"]), device="cuda")
        ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        a = _args(c, x, o_ref, h_ref, flags)
        assert lib.gdn_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), 256, stream) == B.GDN_OK
        o = torch.full_like(o_ref, float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        a = _args(c, x, o, h, flags)
        assert lib.gdn_chunk_fwd_noalloc(ctypes.byref(a), stream) == B.GDN_OK
        assert lib.gdn_check_device_status(None, stream) == B.GDN_OK, f"call {call}: a bounded wait gave up"
        torch.cuda.synchronize()
        assert torch.isfinite(o).all() and torch.isfinite(h).all(), f"call {call}: unwritten outputs"
        assert torch.equal(o, o_ref), f"call {call}: o differs from gdn_chunk_fwd"
        assert torch.equal(h, h_ref), f"call {call}: hT differs from gdn_chunk_fwd"
        if call == 0:   # and against the oracle directly
            oref, href = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, None,
                                                state_qdq=True, w_qdq=True)
            assert rel(o.cpu().double().numpy(), oref) <= TOL_QDQ
            assert rel(h.cpu().double().numpy(), href) <= TOL_QDQ


def test_noalloc_rejects_bad_arguments_before_launch(gdn):
    lib = gdn.load()
    a = B.ChunkArgs(None, None, None, None, None, None, None, None, None, None, 1, 64, 1, 1, 1, 96, 128, 1.0, 0)
    assert lib.gdn_chunk_fwd_noalloc(ctypes.byref(a), None) == B.GDN_ERR_UNSUPPORTED_SHAPE
