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


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq,w_qdq", [(False, False), (True, False), (False, True), (True, True)])
def test_chunked_forward_equals_the_cpp_chunked_oracle(oracle_mod, kda, state_qdq, w_qdq):
    """The chunked-form gradient oracle differentiates the pinned C++ chunked / WY forward (O2),
    W QDQ included: o and hT agree for varlen sequences of 5, 64 and 70 tokens."""
    from oracle.grad import gdn_chunked_grads
    x = workloads.prefill(1, 0, 1, 2, 8, 64, seed=13, kda=kda, h0_std=0.3, seqlens=[5, 64, 70])
    *_, o, hT = gdn_chunked_grads(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=state_qdq,
                                  w_qdq=w_qdq)
    o1, h1 = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=state_qdq,
                                    w_qdq=w_qdq)
    assert rel(o, o1) < 1e-11 and rel(hT, h1) < 1e-11


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq,codec", [(False, "e4m3"), (True, "e4m3"), (True, "int8")])
def test_chunked_gradients_equal_the_recurrent_ones(oracle_mod, kda, state_qdq, codec):
    """Without W QDQ the chunked form is the token recurrence rewritten, and the straight-through
    state quantizer sits at the same 64-token boundaries in both: every gradient agrees (GQA,
    varlen with an empty sequence and one that crosses a boundary)."""
    from oracle.grad import gdn_chunked_grads, gdn_recurrent_grads
    x, do, dhT = tiny(kda, seed=14 + kda, seqlens=[2, 0, 70])
    args = (x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, do, dhT)
    a = gdn_recurrent_grads(*args, kda=kda, state_qdq=state_qdq, codec=codec)
    b = gdn_chunked_grads(*args, kda=kda, state_qdq=state_qdq, codec=codec)
    for name, ga, gb in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0", "o", "hT"), a, b):
        assert rel(gb, ga) < 1e-10, (name, rel(gb, ga))


def test_w_qdq_on_an_exact_tile_changes_no_gradient(oracle_mod):
    """One-token sequences with beta = 1 and g = 0 make W = k; keys of small integers with
    max |k| = 2 give the tile scale 2 / 448, whose codes (k x 224) are all exact E4M3 values, so
    QDQ(W) = W. The straight-through W quantizer then leaves every gradient as it was, which
    pins that it acts on W and nowhere else; random keys show it is active."""
    from oracle.grad import gdn_chunked_grads
    x = workloads.prefill(1, 0, 1, 2, 8, 16, seed=15, h0_std=0.3, seqlens=[1, 1, 1])
    gen = torch.Generator().manual_seed(16)
    keys = torch.randint(-2, 3, x.k.shape, generator=gen).float()
    keys[..., 0] = 2.0                      # every row reaches the tile maximum
    x.beta.fill_(1.0)
    x.g.zero_()
    do = torch.randn((1, 3, 2, 16), generator=gen, dtype=torch.float64)
    dhT = torch.randn((3, 2, 8, 16), generator=gen, dtype=torch.float64)

    def grads(k, w_qdq):
        return gdn_chunked_grads(x.q, k.to(x.k.dtype), x.v, x.g, x.beta, x.h0, x.cu_seqlens, do, dhT, w_qdq=w_qdq)

    exact_on, exact_off = grads(keys, True), grads(keys, False)
    for ga, gb in zip(exact_on, exact_off):
        np.testing.assert_array_equal(ga, gb)
    rand_on, rand_off = grads(x.k.float() * 0.7, True), grads(x.k.float() * 0.7, False)
    assert max(rel(ga, gb) for ga, gb in zip(rand_on[:6], rand_off[:6])) > 1e-4
