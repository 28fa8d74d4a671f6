"""Pins for the fp64 gradient oracle (CPU only).

The gradients are PyTorch autograd through a written-out recurrence with the state QDQ's
backward replaced by the identity ("Torch GDN/KDA decode QAT with INT8 recurrent state",
"Megatron-Core QAT/QAD workflow" step 4: identity straight-through estimator through QDQ). Pinned
by: the forward it differentiates equals the pinned C++ forward oracle; central finite
differences of that forward (no QDQ: smooth) in random directions; and with QDQ, the closed form
of the pure-decay case (beta = 0), where the straight-through gradient of h0 is a sum of decayed
outer products and dq_t is the QDQ'd state times do_t.
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def as_np(x):
    return None if x is None else x.double().numpy()


def tiny(kda, seed, T=6, seqlens=None):
    x = workloads.prefill(1, T, 1, 2, 3, 4, seed=seed, kda=kda, h0_std=0.5, seqlens=seqlens)
    gen = torch.Generator().manual_seed(seed + 100)
    B, TT = x.q.shape[:2]
    N = x.cu_seqlens.numel() - 1 if x.cu_seqlens is not None else B
    do = torch.randn((B, TT, 2, 4), generator=gen, dtype=torch.float64)
    dhT = torch.randn((N, 2, 3, 4), generator=gen, dtype=torch.float64)
    return x, do, dhT


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq", [False, True])
def test_forward_equals_the_cpp_oracle(oracle_mod, kda, state_qdq):
    from oracle.grad import gdn_recurrent_grads
    x = workloads.prefill(1, 0, 1, 2, 8, 64, seed=3, kda=kda, h0_std=0.3, seqlens=[5, 64, 70])
    *_, o, hT = gdn_recurrent_grads(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=state_qdq)
    o1, h1 = oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=state_qdq)
    assert rel(o, o1) < 1e-12 and rel(hT, h1) < 1e-12


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("varlen", [False, True])
def test_finite_differences(oracle_mod, kda, varlen):
    """<grad, E> against the central difference of L = <o, do> + <hT, dhT> along random E, for
    every input (q, k, v, g, beta, h0), GQA (1 q/k head for 2 v-heads), no QDQ."""
    from oracle.grad import gdn_recurrent_grads
    x, do, dhT = tiny(kda, seed=4 + kda, seqlens=[2, 0, 4] if varlen else None)
    names = ("q", "k", "v", "g", "beta", "h0")
    base = {n: getattr(x, n).double() for n in names}
    grads = gdn_recurrent_grads(*(base[n] for n in names[:5]), base["h0"], x.cu_seqlens, do, dhT, kda=kda)[:6]

    def loss(inp):
        *_, o, hT = gdn_recurrent_grads(*(inp[n] for n in names[:5]), inp["h0"], x.cu_seqlens, kda=kda)
        return float((o * do.numpy()).sum() + (hT * dhT.numpy()).sum())

    gen = torch.Generator().manual_seed(9)
    eps = 1e-6
    for i, n in enumerate(names):
        E = torch.randn(base[n].shape, generator=gen, dtype=torch.float64)
        plus, minus = dict(base), dict(base)
        plus[n], minus[n] = base[n] + eps * E, base[n] - eps * E
        fd = (loss(plus) - loss(minus)) / (2 * eps)
        an = float((grads[i] * E.numpy()).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (n, fd, an)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("codec", ["e4m3", "int8"])
def test_straight_through_pure_decay(oracle_mod, kda, codec):
    """beta = 0: S_t = QDQ-at-boundaries of the decayed h0, o_t = S_t^T q_t. With the identity
    backward through QDQ: dh0 = sum_t D_t q_t do_t^T + D_T dhT (D_t the cumulative decay, per key
    row for KDA), dq_t = S_t do_t with S_t the QDQ'd forward state, and dv = 0."""
    from oracle.grad import gdn_recurrent_grads
    T = 150
    x = workloads.prefill(1, T, 1, 1, 8, 64, seed=6, kda=kda, h0_std=0.3)
    x.beta.zero_()
    gen = torch.Generator().manual_seed(7)
    do = torch.randn((1, T, 1, 64), generator=gen, dtype=torch.float64)
    dhT = torch.randn((1, 1, 8, 64), generator=gen, dtype=torch.float64)
    dq, dk, dv, dg, db, dh0, o, hT = gdn_recurrent_grads(x.q, x.k, x.v, x.g, x.beta, x.h0, None, do, dhT, kda=kda,
                                                          state_qdq=True, codec=codec)
    g = as_np(x.g)[0, :, 0]
    q = as_np(x.q)[0, :, 0]
    S = as_np(x.h0)[0, 0].copy()
    D = np.ones(8) if kda else 1.0
    dh0_ref = np.zeros((8, 64))
    qdq = (lambda M: oracle_mod.int8_block_qdq_f64(M, 32)[0]) if codec == "int8" else \
        (lambda M: oracle_mod.tile_qdq_f64(M, 64)[0][0])
    for t in range(T):
        a = np.exp(g[t])
        D = D * a
        S = (a[:, None] if kda else a) * S
        np.testing.assert_allclose(dq[0, t, 0], S @ do[0, t, 0].numpy(), rtol=1e-12, atol=1e-12)
        dh0_ref += (D[:, None] if kda else D) * np.outer(q[t], do[0, t, 0].numpy())
        if (t + 1) % 64 == 0:
            S = qdq(S)
    dh0_ref += (D[:, None] if kda else D) * dhT[0, 0].numpy()
    assert rel(dh0[0, 0], dh0_ref) < 1e-12
    assert not dv.any()
    assert rel(hT[0, 0], S) < 1e-12
