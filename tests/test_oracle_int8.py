"""Pins for the oracle's INT8 block state codec (CPU only).

Reading of the pages (summary of "Torch GDN/KDA decode QAT with INT8 recurrent state": a signed
INT8 state codec whose scales cover blocks of 32 values; "Add experimental GDN/KDA decode and
replay QAT": its tests cover tails of the value axis at codec block sizes 32 and 128): a block is 32 consecutive value columns of one key row
(the last block of a row may be narrower); scale = amax / 127 with the zero guard of the E4M3
tiles; code = nearest integer to x / scale, ties to even, within [-127, 127]; value = code *
scale. Checked by hand-worked blocks (exact scales, every tie), invariants, and the state codec
wired through the recurrence, the chunked form, decode and the handoff.
"""
import numpy as np
import pytest

from fp8_state_qat_gb300 import workloads


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def as_np(x):
    return None if x is None else x.float().numpy().astype(np.float64)


def test_hand_blocks(oracle_mod):
    """amax 127 gives scale 1 exactly, amax 254 scale 2: the quotients are exact, so every
    rounding below is a tie or a plain nearest integer decided by hand."""
    x = np.array([[127.0, -3.5, 2.5, 0.49, -0.5, 126.5, 1.5, -1.5],
                  [254.0, 3.0, -5.0, 1.0, 7.0, -253.0, 0.0, 2.9]], np.float32)
    want = np.array([[127, -4, 2, 0, -0.0, 126, 2, -2],
                     [254, 4, -4, 0, 8, -252, 0, 2]], np.float64)
    for f in (oracle_mod.int8_block_qdq_f32, oracle_mod.int8_block_qdq_f64):
        y, sc = f(x, 8)
        np.testing.assert_array_equal(y, want)
        np.testing.assert_array_equal(sc[:, 0], [1.0, 2.0])
        assert np.signbit(y[0, 4])   # -0.5 rounds to -0


def test_blocks_and_tail(oracle_mod):
    """One scale per 32 columns of a row; a 70-column row has blocks of 32, 32 and 6; rows and
    blocks do not interact."""
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 70)).astype(np.float32)
    x[2, 40] = 50.0   # a large element only moves its own block's scale
    y, sc = oracle_mod.int8_block_qdq_f32(x, 32)
    assert sc.shape == (5, 3)
    for r in range(5):
        for b, (j0, j1) in enumerate(((0, 32), (32, 64), (64, 70))):
            blk = x[r, j0:j1]
            assert sc[r, b] == np.float32(np.abs(blk).max()) / np.float32(127)
            yb, _ = oracle_mod.int8_block_qdq_f32(blk[None], 32)
            np.testing.assert_array_equal(y[r, j0:j1], yb[0])


def test_amax_maps_to_127_and_codes_are_integers(oracle_mod):
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(2000, 32)) * np.exp(rng.normal(size=(2000, 1)) * 3)).astype(np.float32)
    y, sc = oracle_mod.int8_block_qdq_f32(x, 32)
    codes = y.astype(np.float64) / sc.astype(np.float64)   # c * s was rounded to fp32 once
    c = np.round(codes)
    assert np.all(np.abs(codes - c) <= 1e-6 * np.maximum(np.abs(c), 1))
    assert np.abs(c).max() <= 127
    i = np.abs(x).argmax(axis=1)
    np.testing.assert_array_equal(np.abs(c[np.arange(2000), i]), 127)


def test_zero_block_and_idempotence(oracle_mod):
    y, sc = oracle_mod.int8_block_qdq_f32(np.zeros((3, 40), np.float32), 32)
    assert not y.any() and (sc == 1).all()
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5000, 32)).astype(np.float32)
    y1, s1 = oracle_mod.int8_block_qdq_f32(x, 32)
    y2, s2 = oracle_mod.int8_block_qdq_f32(y1, 32)
    np.testing.assert_array_equal(y2, y1)
    np.testing.assert_array_equal(s2, s1)


def test_f64_matches_f32_on_exact_inputs(oracle_mod):
    """Blocks whose quotients are exact in both precisions (amax 127 * 2^k, elements on the grid
    of the scale plus quarter steps) round the same way in fp32 and fp64."""
    rng = np.random.default_rng(4)
    codes = rng.integers(-508, 509, size=(300, 32)) / 4.0
    codes[:, 0] = 127.0
    x = (codes * 2.0 ** rng.integers(-20, 20, size=(300, 1))).astype(np.float32)
    y32, _ = oracle_mod.int8_block_qdq_f32(x, 32)
    y64, _ = oracle_mod.int8_block_qdq_f64(x.astype(np.float64), 32)
    np.testing.assert_array_equal(y32.astype(np.float64), y64)


def small(B=1, T=130, Hqk=1, Hv=1, dk=16, dv=96, seed=0, kda=False, h0_std=0.3, seqlens=None):
    return workloads.prefill(B, T, Hqk, Hv, dk, dv, seed=seed, kda=kda, h0_std=h0_std, seqlens=seqlens)


@pytest.mark.parametrize("kda", [False, True])
def test_state_codec_pure_decay(oracle_mod, kda):
    """beta = 0: S_t = decay^t h0 with the INT8 codec applied (per key row, 32 columns) after
    every 64th token; o_t from the pre-QDQ state."""
    x = small(T=150, dk=8, dv=70, seed=5, kda=kda)
    x.beta.zero_()
    g = as_np(x.g)[0, :, 0]
    S = as_np(x.h0)[0, 0].copy()
    q = as_np(x.q)[0, :, 0]
    o_ref = np.zeros((150, 70))
    for t in range(150):
        S = (np.exp(g[t])[:, None] if kda else np.exp(g[t])) * S
        o_ref[t] = S.T @ q[t]
        if (t + 1) % 64 == 0:
            S = oracle_mod.int8_block_qdq_f64(S, 32)[0]
    for f in (oracle_mod.gdn_recurrent, oracle_mod.gdn_chunked):
        o, hT = f(x.q, x.k, x.v, x.g, x.beta, x.h0, None, kda=kda, state_qdq=True, codec="int8")
        assert rel(o[0, :, 0], o_ref) < 1e-12 and rel(hT[0, 0], S) < 1e-12


@pytest.mark.parametrize("kda", [False, True])
def test_state_codec_chunked_equals_recurrent(oracle_mod, kda):
    x = small(B=1, Hqk=1, Hv=2, dk=32, dv=96, seed=6, kda=kda, seqlens=[0, 1, 64, 65, 130])
    o1, h1 = oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=True,
                                      codec="int8")
    o2, h2 = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=True,
                                    codec="int8")
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12
    oe, he = oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=True)
    assert rel(he, h1) > 1e-4   # the codec changes the result


@pytest.mark.parametrize("kda", [False, True])
def test_state_codec_decode_and_handoff(oracle_mod, kda):
    """Decode with the INT8 codec == the recurrence with a QDQ after every token; the handoff
    == chunked prefix (no state QDQ), INT8 QDQ at the handoff, INT8 decode steps."""
    d = workloads.decode(5, 3, 2, 16, 96, seed=7, kda=kda)
    o, st = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, kda=kda, state_qdq=True, codec="int8")
    tr = lambda t: t.transpose(0, 1).contiguous()
    x = workloads.PrefillInputs(tr(d.q), tr(d.k), tr(d.v), tr(d.g), tr(d.beta), d.state, None, kda=kda)
    o1, h1 = oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, None, kda=kda, state_qdq=True,
                                      qdq_period=1, codec="int8")
    np.testing.assert_array_equal(o, o1.transpose(1, 0, 2, 3))
    np.testing.assert_array_equal(st, h1)
    x = small(T=100, Hv=2, dk=16, dv=64, seed=8, kda=kda)
    o, hT = oracle_mod.gdn_prefill_decode(x.q, x.k, x.v, x.g, x.beta, x.h0, None, [37], kda=kda, state_qdq=True,
                                          codec="int8")
    op, S = oracle_mod.gdn_chunked(x.q[:, :37], x.k[:, :37], x.v[:, :37], x.g[:, :37], x.beta[:, :37], x.h0, None,
                                   kda=kda, state_qdq=False)
    S = oracle_mod.int8_block_qdq_f64(S, 32)[0]
    step = lambda t: t[:, 37:].transpose(0, 1).contiguous()
    od, S = oracle_mod.gdn_decode(step(x.q), step(x.k), step(x.v), step(x.g), step(x.beta), S, kda=kda,
                                  state_qdq=True, codec="int8")
    np.testing.assert_array_equal(o[:, :37], op)
    np.testing.assert_array_equal(o[0, 37:], od[:, 0])
    np.testing.assert_array_equal(hT, S)


def test_rejects_unknown_codec(oracle_mod):
    x = small(T=4, seed=9)
    with pytest.raises(ValueError):
        oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, None, state_qdq=True, codec="int4")
