"""fp8_tile_qdq on the GPU is bit-for-bit the oracle's fp32 tile QDQ ("GDN state/W QAT
foundation", "What does this PR do?": one scale per tile, amax / 448, zero guard, E4M3)."""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bits

pytestmark = pytest.mark.gpu


def wide_inputs(lead, rows, cols, seed):
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-20, 20, (lead, 1, 1)))
    x = (rng.standard_normal((lead, rows, cols)) * mag).astype(np.float32)
    if lead > 2:
        x[1] = 0.0                              # all-zero tiles: scale 1, stay zero
        x[2] = -0.0
    return x


@pytest.mark.parametrize("lead,rows,cols,tile", [
    (64, 128, 128, 64),    # states [dk=128, dv=128]: two tiles each
    (32, 64, 128, 128),    # W tiles [64 x dk]
    (5, 33, 100, 64),      # ragged rows and a narrower last tile
    (16, 128, 256, 64),
    (3, 1, 1, 1),
    (1, 64, 64, 64),
])
def test_qdq_bit_exact(gdn, oracle_mod, lead, rows, cols, tile):
    x = wide_inputs(lead, rows, cols, seed=lead * 7 + cols)
    y, s = gdn.fp8_tile_qdq(torch.from_numpy(x).cuda(), tile)
    yo, so = oracle_mod.tile_qdq_f32(x, tile)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y), bits(yo))
    np.testing.assert_array_equal(bits(s), bits(so))


def test_qdq_rounding_ties_and_saturation(gdn, oracle_mod):
    """Scale exactly 1 (amax = 448): x / s = x, so every E4M3 midpoint is an exact tie; the
    hardware conversion must round it to the even code as the oracle does."""
    grid = [0.0]
    for e in range(-6, 9):
        for m in range(8):
            v = (1 + m / 8) * 2.0 ** e
            if v <= 448:
                grid.append(v)
    grid += [m / 8 * 2.0 ** -6 for m in range(1, 8)]
    grid = np.array(sorted(set(grid)))
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([mids, -mids, grid, np.nextafter(mids, 0), np.nextafter(mids, 1e9)]).astype(np.float32)
    n = vals.size
    cols = 64
    rows = (n + cols - 1) // cols
    x = np.zeros((1, rows, cols), np.float32)
    x.reshape(-1)[:n] = vals
    x[0, -1, -1] = 448.0
    y, s = gdn.fp8_tile_qdq(torch.from_numpy(x).cuda(), cols * 1000)
    yo, so = oracle_mod.tile_qdq_f32(x, cols * 1000)
    assert so[0, 0] == 1.0
    np.testing.assert_array_equal(bits(y), bits(yo))


def test_qdq_denormals_and_in_place(gdn, oracle_mod):
    x = np.zeros((4, 16, 64), np.float32)
    rng = np.random.default_rng(5)
    x[0] = rng.standard_normal((16, 64)) * 1e-39      # fp32 subnormal amax: scale underflows
    x[1] = rng.standard_normal((16, 64)) * 1e-30
    x[2] = np.clip(rng.standard_normal((16, 64)), -3, 3) * 1e38   # near the fp32 maximum, finite
    x[3, 3, 7] = 1e-45
    xt = torch.from_numpy(x).cuda()
    y, s = gdn.fp8_tile_qdq(xt, 64, y=xt)             # in place
    yo, so = oracle_mod.tile_qdq_f32(x, 64)
    np.testing.assert_array_equal(bits(xt), bits(yo))
    np.testing.assert_array_equal(bits(s), bits(so))


def test_qdq_empty(gdn):
    x = torch.zeros((0, 8, 64), device="cuda")
    y, s = gdn.fp8_tile_qdq(x, 64)
    assert y.shape == (0, 8, 64) and s.shape == (0, 1)
    x = torch.zeros((2, 0, 64), device="cuda")
    y, s = gdn.fp8_tile_qdq(x, 64)
    torch.cuda.synchronize()
    assert (s.cpu() == 1.0).all()


def test_quotient_matches_ieee_divide_over_all_significands(gdn):
    """The standalone QDQ ops divide by the tile scale as the rounded reciprocal plus two FMA
    corrections (common.cuh). Against __fdiv_rn, bit for bit, over (1) every fp32 significand of
    x at 22 binades (x / s from 2^-13 to 2^10: every E4M3 binade, subnormal codes and saturation)
    times 256 scale significands, and (2) every significand of s at 4 binades times 256 values of
    x: the quotient bits, hence the E4M3 codes, must all agree; the paired instruction form must
    agree with the scalar one. The fused kernels' plain reciprocal product is counted for
    reference only."""
    import native
    from helpers import record
    lib = native.load()
    fn = lib.gdnqat_testing_quotient_sweep
    fn.restype = ctypes.c_int
    rng = np.random.default_rng(11)
    sig = lambda n: (1.0 + rng.integers(0, 1 << 23, n) / float(1 << 23)).astype(np.float32)
    scales = np.concatenate([np.float32([1.0, np.nextafter(np.float32(1), np.float32(2)),
                                         np.nextafter(np.float32(2), np.float32(1))]), sig(253)])
    xs = sig(256) * np.float32(2.0) ** rng.integers(-12, 10, 256).astype(np.float32)
    xs[::2] *= -1
    for mode, vals, exps in ((0, scales, np.arange(-12, 10)), (1, xs, np.array([-3, 0, 5, 20]))):
        dv = torch.from_numpy(np.ascontiguousarray(vals, np.float32)).cuda()
        de = torch.from_numpy(exps.astype(np.int32)).cuda()
        counts = torch.zeros(4, dtype=torch.int64, device="cuda")
        first = torch.zeros(3, dtype=torch.int32, device="cuda")
        rc = fn(ctypes.c_void_p(dv.data_ptr()), len(vals), ctypes.c_void_p(de.data_ptr()), len(exps), mode,
                ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(first.data_ptr()), None)
        assert rc == 0
        torch.cuda.synchronize()
        c = counts.cpu().tolist()
        f = first.cpu().numpy().view(np.uint32)
        record("plain_reciprocal_code_mismatches", c[3], mode=mode, pairs=(1 << 23) * len(vals) * len(exps))
        assert c[0] == 0 and c[1] == 0, (mode, c, f[:2].view(np.float32))
        assert c[2] == 0, (mode, c)


def test_tile_scale_matches_ieee_divide_for_every_amax(gdn):
    """The tile scale amax / 448 (zero guard: 1) every QDQ site uses is computed as the rounded
    reciprocal of 448 plus two FMA corrections; over every non-negative finite fp32 amax it must
    equal the IEEE round-to-nearest divide bit for bit."""
    import native
    lib = native.load()
    fn = lib.gdnqat_testing_scale_sweep
    fn.restype = ctypes.c_int
    counts = torch.zeros(1, dtype=torch.int64, device="cuda")
    first = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fn(ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(first.data_ptr()), None) == 0
    torch.cuda.synchronize()
    assert int(counts.item()) == 0, (int(counts.item()), hex(int(first.item()) & 0xffffffff))
