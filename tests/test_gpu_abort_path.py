"""The bounded waits' give-up path, driven on purpose and without a fault.

The test-only library compiles the two-kernel chunk forward with GDN_WAIT_LIMIT = 0: every
pipeline mbarrier wait of the prep and chain kernels gives up on its first poll. Each CTA then
raises its abort flag, leaves its loops at the next checked barrier without issuing more MMAs or
copies, sets the workspace status word, waits for the TMA loads already in flight with their
own limits, frees its TMEM and exits ("GDN state/W QAT foundation", "What does this PR do?":
failures are reported as explicit errors, never as a hang). The product library must then report
GDN_ERR_DEVICE_TIMEOUT for that workspace, and its next regular call on the same device must
be correct."""
import ctypes

import pytest
import torch

import native
from fp8_state_qat_gb300 import gdnqat as B
from fp8_state_qat_gb300 import workloads
from helpers import TOL_QDQ, rel

pytestmark = pytest.mark.gpu


def test_short_waits_report_timeout_and_device_stays_usable(gdn, oracle_mod):
    lib, tlib = gdn.load(), native.load()
    tlib.gdnqat_testing_split_fwd.restype = ctypes.c_int
    tlib.gdnqat_testing_split_fwd.argtypes = [ctypes.POINTER(B.ChunkArgs), ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]
    x = workloads.prefill(1, 256, 2, 2, 128, 128, seed=91, h0_std=0.1)
    c = {k: getattr(x, k).cuda() for k in ("q", "k", "v", "g", "beta", "h0")}
    s = x.shape
    flags = B.GDN_FLAG_STATE_QDQ | B.GDN_FLAG_W_QDQ
    o = torch.zeros((s["B"], s["T"], s["Hv"], s["dv"]), device="cuda")
    h = torch.zeros((s["N"], s["Hv"], s["dk"], s["dv"]), device="cuda")
    a = B.ChunkArgs(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["g"].data_ptr(),
                    c["beta"].data_ptr(), c["h0"].data_ptr(), None, None, o.data_ptr(), h.data_ptr(),
                    s["B"], s["T"], s["N"], s["Hqk"], s["Hv"], s["dk"], s["dv"], 1.0, flags)
    nbytes = lib.gdn_chunk_fwd_workspace_size(ctypes.byref(a))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert tlib.gdnqat_testing_split_fwd(ctypes.byref(a), ws.data_ptr(), nbytes, stream) == 0
    assert lib.gdn_check_device_status(ctypes.c_void_p(ws.data_ptr()), stream) == B.GDN_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()   # no sticky CUDA error: the kernels returned normally

    # the same workspace and device, the regular library: correct results, status clear
    assert lib.gdn_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), nbytes, stream) == B.GDN_OK
    assert lib.gdn_check_device_status(ctypes.c_void_p(ws.data_ptr()), stream) == B.GDN_OK
    oref, href = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, None, state_qdq=True, w_qdq=True)
    assert rel(o.cpu().double().numpy(), oref) <= TOL_QDQ
    assert rel(h.cpu().double().numpy(), href) <= TOL_QDQ
