"""Pins for the oracle's E4M3 rounding and tile QDQ (CPU only).

The QDQ contract ("GDN state/W QAT foundation", "What does this PR do?"): dynamic FP8
E4M3 (num_bits (4,3)), one scalar scale per tile, scale = amax / 448 (1 for an all-zero tile),
x -> E4M3(x / scale) * scale. Every check here reaches the oracle's answer by another
route: decoding the 256 bit patterns, brute-force nearest search, torch's own float8 cast,
hand-worked values, and invariants (amax element -> +-448, zero tile, idempotence).
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def e4m3_decode_all():
    """All 256 E4M3 (fn) bit patterns decoded from the bit layout: s eeee mmm, bias 7,
    exponent field 0 = subnormal (m/8 * 2^-6), pattern s.1111.111 = NaN, no infinities."""
    vals = {}
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            continue  # NaN
        if e == 0:
            v = s * (m / 8.0) * 2.0 ** -6
        else:
            v = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = v
    return vals


def brute_nearest(y, grid_pos):
    """Nearest finite E4M3 value by exhaustive search; ties to the code with even mantissa;
    magnitudes beyond 448 saturate."""
    a = abs(y)
    if a >= 448.0:
        return np.copysign(448.0, y)
    best = None
    for code, v in grid_pos:
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0):
            best = (d, v, code)
    return np.copysign(best[1], y)


@pytest.fixture(scope="module")
def grid():
    vals = e4m3_decode_all()
    return sorted(((c, v) for c, v in vals.items() if v >= 0 and not (c & 0x80)), key=lambda t: t[1])


def test_e4m3_code_table(oracle_mod):
    vals = e4m3_decode_all()
    assert len(vals) == 254
    finite = sorted(set(vals.values()))
    assert max(finite) == 448.0 and min(finite) == -448.0
    assert min(v for v in finite if v > 0) == 2.0 ** -9
    for v in finite:  # every grid point is a fixed point of the rounding
        assert oracle_mod.e4m3_rne(v) == v


def test_e4m3_brute_force(oracle_mod, grid):
    rng = np.random.default_rng(11)
    ys = np.concatenate([
        rng.uniform(-500, 500, 3000),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),      # subnormal neighbourhood
        np.exp(rng.uniform(np.log(1e-4), np.log(460), 3000)) * rng.choice([-1, 1], 3000),
    ])
    for y in ys:
        assert oracle_mod.e4m3_rne(float(y)) == brute_nearest(float(y), grid), y


def test_e4m3_midpoints_tie_to_even(oracle_mod, grid):
    for (c0, v0), (c1, v1) in zip(grid[:-1], grid[1:]):
        mid = (v0 + v1) / 2.0
        want = v0 if (c0 & 1) == 0 else v1
        assert oracle_mod.e4m3_rne(mid) == want
        assert oracle_mod.e4m3_rne(-mid) == -want
    # past the largest finite value: satfinite
    for y in (448.0, 460.0, 464.0, 470.0, 1e6):
        assert oracle_mod.e4m3_rne(y) == 448.0 and oracle_mod.e4m3_rne(-y) == -448.0


def test_e4m3_matches_torch_cast(oracle_mod):
    """torch's float8_e4m3fn cast rounds to nearest-even but does not saturate, so compare
    below 448 only."""
    rng = np.random.default_rng(12)
    ys = np.concatenate([rng.uniform(-447.9, 447.9, 20000).astype(np.float32),
                         (rng.standard_normal(20000) * 0.01).astype(np.float32)])
    t = torch.from_numpy(ys).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    mine = np.array([oracle_mod.e4m3_rne(float(y)) for y in ys])
    np.testing.assert_array_equal(mine, t.astype(np.float64))


def test_qdq_hand_example(oracle_mod):
    ex = json.load(open(GOLDEN))["qdq_tile_2x2"]
    x = np.array(ex["x"], np.float64)
    y, s = oracle_mod.tile_qdq_f64(x, 64)
    assert s[0, 0] == pytest.approx(ex["scale"], rel=1e-15)
    np.testing.assert_allclose(y[0], np.array(ex["y"]), rtol=1e-15)
    yf, sf = oracle_mod.tile_qdq_f32(x.astype(np.float32), 64)
    np.testing.assert_allclose(yf[0], np.array(ex["y"]), rtol=1e-6)
    np.testing.assert_allclose(yf[0] / sf[0, 0], np.array(ex["codes"], np.float64), rtol=1e-6)


def _random_tiles(rng, lead, rows, cols):
    scale = np.exp(rng.uniform(-12, 12, (lead, 1, 1)))
    return (rng.standard_normal((lead, rows, cols)) * scale).astype(np.float32)


def test_qdq_amax_element_maps_to_448(oracle_mod, grid):
    rng = np.random.default_rng(13)
    x = _random_tiles(rng, 2000, 16, 64)
    y, s = oracle_mod.tile_qdq_f32(x, 64)
    for l in range(x.shape[0]):
        i = np.unravel_index(np.argmax(np.abs(x[l])), x[l].shape)
        sc = np.float32(s[l, 0])
        assert sc == np.float32(np.float32(np.max(np.abs(x[l]))) / np.float32(448.0))
        assert y[l][i] == np.float32(np.float32(448.0) * sc) * np.sign(x[l][i])
    # every dequantized value is fl32(code * scale) with code on the E4M3 grid, |code| <= 448
    codes = np.abs(y.astype(np.float64) / s[:, :, None].astype(np.float64)).reshape(-1)
    g = np.array(sorted({v for _, v in grid}))
    idx = np.clip(np.searchsorted(g, codes), 1, len(g) - 1)
    nearest = np.where(codes - g[idx - 1] < g[idx] - codes, g[idx - 1], g[idx])
    assert np.all(np.abs(codes - nearest) <= 2.0 ** -23 * nearest)
    assert codes.max() <= 448.0 * (1 + 2.0 ** -23)


def test_qdq_zero_tile(oracle_mod):
    x = np.zeros((3, 8, 70), np.float32)
    x[1, 2, 5] = 1.5   # a nonzero in tile 0 of lead 1 only
    y, s = oracle_mod.tile_qdq_f32(x, 64)
    assert s.shape == (3, 2)
    assert (s[0] == 1.0).all() and (s[2] == 1.0).all() and s[1, 1] == 1.0
    assert s[1, 0] == np.float32(np.float32(1.5) / np.float32(448.0))
    np.testing.assert_array_equal(y[0], 0.0)
    np.testing.assert_array_equal(y[2], 0.0)
    assert y[1, 2, 5] == np.float32(1.5)


def test_qdq_tiles_are_independent(oracle_mod):
    """A [rows, cols] matrix with tile width 64 equals QDQ of each column block alone,
    including a ragged last block (cols = 100 -> 64 + 36)."""
    rng = np.random.default_rng(14)
    x = _random_tiles(rng, 4, 32, 100)
    x[:, :, 64:] *= 1000.0
    y, s = oracle_mod.tile_qdq_f32(x, 64)
    ya, sa = oracle_mod.tile_qdq_f32(np.ascontiguousarray(x[:, :, :64]), 64)
    yb, sb = oracle_mod.tile_qdq_f32(np.ascontiguousarray(x[:, :, 64:]), 64)
    np.testing.assert_array_equal(y[:, :, :64], ya)
    np.testing.assert_array_equal(y[:, :, 64:], yb)
    np.testing.assert_array_equal(s, np.concatenate([sa, sb], axis=1))


def test_qdq_idempotent(oracle_mod):
    rng = np.random.default_rng(15)
    x = _random_tiles(rng, 5000, 8, 64)
    y1, s1 = oracle_mod.tile_qdq_f32(x, 64)
    y2, s2 = oracle_mod.tile_qdq_f32(y1, 64)
    np.testing.assert_array_equal(y1.view(np.uint32), y2.view(np.uint32))
    np.testing.assert_array_equal(s1, s2)


def test_qdq_scale_fixed_point_all_amax_in_one_binade():
    """Idempotence needs fl(fl(448 s) / 448) == s for s = fl(amax / 448). Sweep every fp32
    amax in [1, 2); the relation is invariant under scaling by powers of two (normal range)."""
    a = (np.arange(2 ** 23, dtype=np.uint32) + np.uint32(0x3F800000)).view(np.float32)
    s = (a / np.float32(448.0)).astype(np.float32)
    back = ((np.float32(448.0) * s).astype(np.float32) / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(back, s)


def test_qdq_f64_matches_f32_on_exact_inputs(oracle_mod):
    """Where the fp32 steps are exact (power-of-two amax, values already on the grid)
    the fp64 and fp32 versions agree exactly."""
    rng = np.random.default_rng(16)
    codes = rng.choice([-448, -224, -3.5, -0.25, 0.0, 0.125, 1.0, 13.0, 96.0, 448.0], (10, 8, 64))
    codes[:, 0, 0] = 448.0   # every tile's amax is a power-of-two multiple of 448
    x = (codes * 2.0 ** -5).astype(np.float32)
    y32, _ = oracle_mod.tile_qdq_f32(x, 64)
    y64, _ = oracle_mod.tile_qdq_f64(x.astype(np.float64), 64)
    np.testing.assert_array_equal(y32.astype(np.float64), y64)
    np.testing.assert_array_equal(y64, x.astype(np.float64))
