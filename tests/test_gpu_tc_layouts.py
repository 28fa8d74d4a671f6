"""Hardware check of the tensor-core operand layouts the chunked forward relies on: a
tcgen05 MMA on bf16 / tf32 operands staged in the 128-byte-swizzled K-major or MN-major
shared-memory layout must reproduce a CPU matrix product of the same rounded operands."""
import ctypes

import numpy as np
import pytest
import torch

import native

pytestmark = pytest.mark.gpu


def rounded(x, kind):
    t = torch.from_numpy(x)
    if kind == 0:
        return t.to(torch.bfloat16).double().numpy()
    u = t.view(torch.int32).numpy().astype(np.int64)
    r = ((u + 0x1000) >> 13) << 13          # round to nearest, ties away, 10 mantissa bits
    return r.astype(np.int32).view(np.float32).astype(np.float64)


# (kind, a_mn, b_mn): bf16 in every major combination, tf32 K-major only -- the chunked
# forward stages tf32 operands K-major (an MN-major tf32 operand needs a different swizzle
# mode than the 128-byte one staged here).
COMBOS = [(0, 0, 0), (0, 0, 1), (0, 1, 0), (0, 1, 1), (1, 0, 0)]


@pytest.mark.parametrize("kind,a_mn,b_mn", COMBOS)
@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("M", [128, 64])
def test_mma_layouts(gdn, kind, a_mn, b_mn, N, K, M):
    """M = 128: row m of D in TMEM lane m. M = 64: row m in lane 32 (m / 16) + m % 16."""
    fn = native.load().gdnqat_internal_tc_selftest
    fn.restype = ctypes.c_int
    rng = np.random.default_rng(kind * 8 + a_mn * 4 + b_mn * 2 + N + K)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dD = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.c_void_p(dA.data_ptr()), ctypes.c_void_p(dB.data_ptr()), ctypes.c_void_p(dD.data_ptr()), None,
            M, N, K, kind, a_mn, b_mn, ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "bounded wait gave up"
    want = rounded(A, kind) @ rounded(B, kind)
    got = dD.cpu().double().numpy()
    if M == 64:
        got = got[[32 * (m // 16) + m % 16 for m in range(64)]]
    np.testing.assert_allclose(got, want, rtol=1e-4, atol=1e-4 * np.abs(want).max())


@pytest.mark.parametrize("N", [64, 128])
def test_tmem_16x32bx2_reads_m64_rows(gdn, N):
    """The 16-lane two-half TMEM load on an M = 64 accumulator: thread t of warp w reads row
    16 w + t % 16, columns [c0 + (t / 16) N / 2, + 16). Every row of the product is recovered and
    lanes 16-31 of each quadrant are never touched."""
    fn = native.load().gdnqat_internal_tc_selftest
    fn.restype = ctypes.c_int
    M, K = 64, 128
    rng = np.random.default_rng(500 + N)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dD = torch.full((128, N), float("nan"), device="cuda")
    dD2 = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.c_void_p(dA.data_ptr()), ctypes.c_void_p(dB.data_ptr()), ctypes.c_void_p(dD.data_ptr()),
            ctypes.c_void_p(dD2.data_ptr()), M, N, K, 0, 0, 0, ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "bounded wait gave up"
    want = rounded(A, 0) @ rounded(B, 0)
    got = dD2.cpu().double().numpy()
    rows = [32 * (m // 16) + m % 16 for m in range(64)]
    np.testing.assert_allclose(got[rows], want, rtol=1e-4, atol=1e-4 * np.abs(want).max())
    untouched = [l for l in range(128) if l not in rows]
    assert np.isnan(got[untouched]).all()


@pytest.mark.parametrize("N", [64, 128])
def test_tmem_16x32bx2_upper_half_lanes_m128(gdn, N):
    """An M = 128 accumulator read with the 16-lane two-half shape at lane offsets 0 and 16 of
    each quadrant: every row comes back (the chain kernel reads X from lanes 0-15 and Y from
    lanes 16-31 of one M = 128 product whose A rows interleave W and Q in 16-row groups)."""
    fn = native.load().gdnqat_internal_tc_selftest
    fn.restype = ctypes.c_int
    M, K = 128, 128
    rng = np.random.default_rng(600 + N)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dD = torch.full((128, N), float("nan"), device="cuda")
    dD2 = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.c_void_p(dA.data_ptr()), ctypes.c_void_p(dB.data_ptr()), ctypes.c_void_p(dD.data_ptr()),
            ctypes.c_void_p(dD2.data_ptr()), M, N, K, 0, 0, 0, ctypes.c_void_p(st.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "bounded wait gave up"
    want = rounded(A, 0) @ rounded(B, 0)
    np.testing.assert_allclose(dD2.cpu().double().numpy(), want, rtol=1e-4, atol=1e-4 * np.abs(want).max())
