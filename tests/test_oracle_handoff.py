"""Pins for the oracle's prefill -> decode handoff (CPU only).

The schedule is the one of "Torch GDN/KDA decode QAT with INT8 recurrent state", section
"Megatron-Core QAT/QAD workflow", steps 2-3 (and its "Ordinary state-QDQ path" flowchart): a
sequence's first prefill_lengths[n] tokens run as chunked prefill whose state is not quantized
inside the prefix; if tokens remain, the state is QDQ'd once at the hand-over, and every remaining
token (teacher forced: the sequence's own tokens) is a decode step that stores a QDQ'd state.

Each check reaches the answer by another route: the plain recurrence without any QDQ (the
schedule cannot matter without quantization), a brute-force two-token example written out with
numpy, and the composition of the separately pinned chunked prefill, tile QDQ and decode step.
"""
import numpy as np
import pytest

from fp8_state_qat_gb300 import workloads


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def as_np(x):
    return None if x is None else x.float().numpy().astype(np.float64)


def small(B=1, T=130, Hqk=1, Hv=1, dk=16, dv=16, seed=0, kda=False, h0_std=0.3, seqlens=None):
    return workloads.prefill(B, T, Hqk, Hv, dk, dv, seed=seed, kda=kda, h0_std=h0_std, seqlens=seqlens)


def handoff(o, x, P, **kw):
    return o.gdn_prefill_decode(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, P, kda=x.kda, **kw)


def composed(o, x, P, state_qdq, w_qdq):
    """Chunked prefix (no state QDQ) -> tile QDQ of the handed-off state -> decode steps, run
    sequence by sequence through the separately pinned oracle functions."""
    B, T = x.q.shape[:2]
    Hv, dk, dv = x.v.shape[2], x.q.shape[3], x.v.shape[3]
    cu = x.cu_seqlens.tolist() if x.cu_seqlens is not None else [n * T for n in range(B + 1)]
    N = len(cu) - 1
    flat = lambda t: t.reshape(1, B * T, *t.shape[2:])
    q, k, v, g, beta = (flat(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    h0 = as_np(x.h0) if x.h0 is not None else np.zeros((N, Hv, dk, dv))
    o_all = np.zeros((1, B * T, Hv, dv))
    hT_all = np.zeros((N, Hv, dk, dv))
    for n in range(N):
        a, L, p = cu[n], cu[n + 1] - cu[n], P[n]
        sp = slice(a, a + p)
        op, S = o.gdn_chunked(q[:, sp], k[:, sp], v[:, sp], g[:, sp], beta[:, sp], h0[n:n + 1], None, kda=x.kda,
                              state_qdq=False, w_qdq=w_qdq)
        o_all[:, sp] = op
        if p < L:
            if state_qdq:
                S = o.tile_qdq_f64(S.reshape(Hv, dk, dv), 64)[0].reshape(1, Hv, dk, dv)
            ss = slice(a + p, a + L)
            step = lambda t: t[:, ss].transpose(0, 1).contiguous()   # tokens as decode steps, N = 1
            od, S = o.gdn_decode(step(q), step(k), step(v), step(g), step(beta), S, kda=x.kda, state_qdq=state_qdq)
            o_all[0, ss] = od[:, 0]
        hT_all[n] = S[0]
    return o_all.reshape(B, T, Hv, dv), hT_all


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("w_qdq", [False, True])
def test_equals_composition_of_pinned_parts(oracle_mod, kda, w_qdq):
    lens = [0, 1, 5, 64, 100, 128, 130, 200]
    P = [0, 0, 5, 64, 37, 64, 130, 63]
    x = small(Hqk=1, Hv=2, dk=32, dv=96, seed=21, kda=kda, seqlens=lens)
    for state_qdq in (False, True):
        o, hT = handoff(oracle_mod, x, P, state_qdq=state_qdq, w_qdq=w_qdq)
        oc, hc = composed(oracle_mod, x, P, state_qdq, w_qdq)
        np.testing.assert_array_equal(o, oc)
        np.testing.assert_array_equal(hT, hc)


def test_dense_batch_equals_composition(oracle_mod):
    x = small(B=3, T=128, Hqk=1, Hv=2, dk=16, dv=64, seed=22)
    P = [64, 0, 128]
    o, hT = handoff(oracle_mod, x, P, state_qdq=True, w_qdq=True)
    oc, hc = composed(oracle_mod, x, P, True, True)
    np.testing.assert_array_equal(o, oc)
    np.testing.assert_array_equal(hT, hc)


@pytest.mark.parametrize("kda", [False, True])
def test_without_quantizers_equals_plain_recurrence(oracle_mod, kda):
    """With both quantizers off the prefix/suffix split changes nothing but rounding."""
    lens = [7, 64, 150]
    x = small(Hqk=1, Hv=2, dk=32, dv=64, seed=23, kda=kda, seqlens=lens)
    o1, h1 = oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=False)
    for P in ([0, 0, 0], [7, 64, 150], [3, 32, 100]):
        o, hT = handoff(oracle_mod, x, P, state_qdq=False, w_qdq=False)
        assert rel(o, o1) < 1e-12 and rel(hT, h1) < 1e-12


def test_two_tokens_by_hand(oracle_mod):
    """T = 2, prefix 1: S1 = a1 h0 + b1 k1 (v1 - a1 h0^T k1)^T (chunked, no QDQ), o1 = S1^T q1;
    then S1 <- QDQ(S1); S2 = a2 S1 + b2 k2 (v2 - a2 S1^T k2)^T, o2 = S2^T q2, S2 <- QDQ(S2)."""
    x = small(T=2, dk=2, dv=3, seed=24)
    q, k, v = as_np(x.q)[0, :, 0], as_np(x.k)[0, :, 0], as_np(x.v)[0, :, 0]
    a = np.exp(as_np(x.g)[0, :, 0])
    b = as_np(x.beta)[0, :, 0]
    S = as_np(x.h0)[0, 0]
    qdq = lambda M: oracle_mod.tile_qdq_f64(M, 64)[0][0]
    S1 = a[0] * S + b[0] * np.outer(k[0], v[0] - a[0] * S.T @ k[0])
    o1 = S1.T @ q[0]
    S1 = qdq(S1)
    S2 = a[1] * S1 + b[1] * np.outer(k[1], v[1] - a[1] * S1.T @ k[1])
    o2 = S2.T @ q[1]
    S2 = qdq(S2)
    o, hT = handoff(oracle_mod, x, [1], state_qdq=True)
    assert rel(o[0, 0, 0], o1) < 1e-12 and rel(o[0, 1, 0], o2) < 1e-12
    assert rel(hT[0, 0], S2) < 1e-12


def test_handoff_state_is_quantized_only_with_a_suffix(oracle_mod):
    x = small(T=64, dk=16, dv=64, seed=25)
    _, h_full = handoff(oracle_mod, x, [64], state_qdq=True)        # no suffix: plain prefill state
    _, h_plain = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, None, state_qdq=False)
    np.testing.assert_array_equal(h_full, h_plain)
    assert not np.array_equal(oracle_mod.tile_qdq_f64(h_full[0, 0], 64)[0][0], h_full[0, 0])   # not QDQ'd


def test_rejects_bad_prefill_lengths(oracle_mod):
    x = small(T=10, seed=26)
    with pytest.raises(ValueError):
        handoff(oracle_mod, x, [11])
    with pytest.raises(ValueError):
        handoff(oracle_mod, x, [-1])
