"""Pins for the oracle's recurrence (O1), chunked/WY form (O2) and decode step (CPU only).

Each check reaches the oracle's answer by a route other than the oracle's own loops:
hand-worked examples (tests/golden/hand_examples.json), the closed product form of the
recurrence, closed forms for beta = 0 (pure decay) and for alpha = beta = 1 with
orthonormal keys (exact overwrite), a closed form for W QDQ, split/resume, varlen ==
per-sequence runs, GQA == materialised head repeat, KDA with equal channels == GDN, and
O1 == O2.

Sources: state QDQ at every 64-token boundary with one scale per full-key x 64-value-
column tile ("GDN state/W QAT foundation", "What does this PR do?"); decode order
("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD workflow",
step 3); KDA per-key-channel retention ("Add KDA prefill numerical emulation for QAT",
"What does this PR do?").
"""
import json
import os

import numpy as np
import pytest

from fp8_state_qat_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


def as_np(x):
    return None if x is None else x.float().numpy().astype(np.float64)


def small(B=1, T=130, Hqk=1, Hv=1, dk=16, dv=16, seed=0, kda=False, h0_std=0.3, seqlens=None):
    return workloads.prefill(B, T, Hqk, Hv, dk, dv, seed=seed, kda=kda, h0_std=h0_std, seqlens=seqlens)


def run1(o, x, **kw):
    return o.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=x.kda, **kw)


def run2(o, x, **kw):
    return o.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=x.kda, **kw)


# --- hand-worked examples ---------------------------------------------------------------

def _hand_inputs(ex, kda):
    T = len(ex["beta"])
    q = np.array(ex["q"], np.float32).reshape(1, T, 1, -1)
    k = np.array(ex["k"], np.float32).reshape(1, T, 1, -1)
    v = np.array(ex["v"], np.float32).reshape(1, T, 1, -1)
    beta = np.array(ex["beta"], np.float32).reshape(1, T, 1)
    alpha = np.array(ex["alpha"], np.float64)
    g = np.log(alpha).astype(np.float32).reshape((1, T, 1, -1) if kda else (1, T, 1))
    h0 = np.array(ex["h0"], np.float64).reshape(1, 1, 2, 2)
    return q, k, v, g, beta, h0


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_hand_example_gdn(oracle_mod, form):
    ex = json.load(open(GOLDEN))["gdn_two_tokens"]
    q, k, v, g, beta, h0 = _hand_inputs(ex, kda=False)
    f = oracle_mod.gdn_recurrent if form == "recurrent" else oracle_mod.gdn_chunked
    o, hT = f(q, k, v, g, beta, h0)
    np.testing.assert_allclose(o.reshape(2, 2), np.array(ex["o"]), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(hT.reshape(2, 2), np.array(ex["hT"]), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_hand_example_kda(oracle_mod, form):
    ex = json.load(open(GOLDEN))["kda_one_token"]
    q, k, v, g, beta, h0 = _hand_inputs(ex, kda=True)
    f = oracle_mod.gdn_recurrent if form == "recurrent" else oracle_mod.gdn_chunked
    o, hT = f(q, k, v, g, beta, h0, kda=True)
    np.testing.assert_allclose(o.reshape(1, 2), np.array(ex["o"]), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(hT.reshape(2, 2), np.array(ex["hT"]), rtol=1e-6, atol=1e-6)


def test_hand_example_decode_qdq(oracle_mod):
    ex = json.load(open(GOLDEN))["decode_qdq_one_token"]
    q = np.array(ex["q"], np.float32).reshape(1, 1, 1, 2)
    k = np.array(ex["k"], np.float32).reshape(1, 1, 1, 2)
    v = np.array(ex["v"], np.float32).reshape(1, 1, 1, 2)
    g = np.log(np.array([ex["alpha"]], np.float64)).astype(np.float32).reshape(1, 1, 1)
    beta = np.array([ex["beta"]], np.float32).reshape(1, 1, 1)
    st = np.array(ex["h0"], np.float64).reshape(1, 1, 2, 2)
    o, st2 = oracle_mod.gdn_decode(q, k, v, g, beta, st, state_qdq=True)
    np.testing.assert_allclose(o.reshape(2), np.array(ex["o"]), rtol=1e-6)
    np.testing.assert_allclose(st2.reshape(2, 2), np.array(ex["state_after"]), rtol=1e-6)


# --- closed product form (brute force on tiny problems) ---------------------------------

@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("dk,dv,T", [(2, 2, 1), (2, 2, 3), (3, 2, 5), (4, 3, 5)])
def test_product_form(oracle_mod, kda, dk, dv, T):
    """S_t = M_t S_{t-1} + b_t k_t v_t^T with M_t = (I - b_t k_t k_t^T) Diag(a_t): the
    transition matrices multiplied out in closed form."""
    x = small(T=T, dk=dk, dv=dv, seed=7 + T, kda=kda)
    q, k, v, g, beta, h0 = (as_np(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    Ms, Bs = [], []
    for t in range(T):
        a = np.exp(g[0, t, 0]) * np.ones(dk) if not kda else np.exp(g[0, t, 0])
        kt = k[0, t, 0]
        Ms.append((np.eye(dk) - beta[0, t, 0] * np.outer(kt, kt)) @ np.diag(a))
        Bs.append(beta[0, t, 0] * np.outer(kt, v[0, t, 0]))
    o_ref = np.zeros((T, dv))
    for t in range(T):
        prod = np.eye(dk)
        S = np.zeros((dk, dv))
        for j in range(t, -1, -1):           # S_t = sum_j (M_t..M_{j+1}) B_j + (M_t..M_1) h0
            S += prod @ Bs[j]
            prod = prod @ Ms[j]
        S += prod @ h0[0, 0]
        o_ref[t] = S.T @ q[0, t, 0]
    o1, h1 = run1(oracle_mod, x)
    o2, h2 = run2(oracle_mod, x, chunk=64)
    np.testing.assert_allclose(o1[0, :, 0], o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h1[0, 0], S, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o2[0, :, 0], o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h2[0, 0], S, rtol=1e-12, atol=1e-13)


# --- O1 == O2 ---------------------------------------------------------------------------

@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("state_qdq", [False, True])
def test_recurrent_equals_chunked(oracle_mod, kda, chunk, state_qdq):
    x = small(B=2, T=200, Hqk=1, Hv=2, dk=32, dv=80, seed=chunk + 3 * kda, kda=kda)
    o1, h1 = run1(oracle_mod, x, state_qdq=state_qdq)
    o2, h2 = run2(oracle_mod, x, chunk=chunk, state_qdq=state_qdq)
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


def test_recurrent_equals_chunked_varlen_gqa(oracle_mod):
    x = small(B=1, Hqk=2, Hv=4, dk=32, dv=64, seed=5, seqlens=[1, 63, 64, 65, 0, 129])
    for sq in (False, True):
        o1, h1 = run1(oracle_mod, x, state_qdq=sq)
        o2, h2 = run2(oracle_mod, x, state_qdq=sq)
        assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


# --- beta = 0: pure decay -----------------------------------------------------------------

@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq", [False, True])
def test_pure_decay(oracle_mod, kda, state_qdq):
    # KDA + QDQ runs one boundary only: past the first QDQ, elements in the same key row as
    # the new amax keep exact code ratios under pure decay, so x / scale can land exactly on
    # an E4M3 midpoint (e.g. 336 between 320 and 352) and fp64 rounding order picks the side.
    T, dk, dv = (100 if (kda and state_qdq) else 200), 16, 128
    x = small(T=T, dk=dk, dv=dv, seed=21, kda=kda)
    x.beta.zero_()
    q, g, h0 = as_np(x.q)[0, :, 0], as_np(x.g)[0, :, 0], as_np(x.h0)[0, 0]
    gc = g if kda else np.repeat(g[:, None], dk, axis=1)        # [T, dk]
    o_ref = np.zeros((T, dv))
    S_base, base_t = h0.copy(), 0                                # state at the last boundary
    for t in range(T):
        decay = np.exp(np.sum(gc[base_t:t + 1], axis=0))         # exp(gamma_t - gamma_base)
        S_t = decay[:, None] * S_base
        o_ref[t] = S_t.T @ q[t]
        if state_qdq and (t + 1) % 64 == 0:
            S_t = oracle_mod.tile_qdq_f64(S_t, 64)[0][0]
            S_base, base_t = S_t, t + 1
    for f in (run1, run2):
        o, hT = f(oracle_mod, x, state_qdq=state_qdq)
        assert rel(o[0, :, 0], o_ref) < 1e-12
        assert rel(hT[0, 0], S_t) < 1e-12


# --- alpha = beta = 1 with orthonormal keys: exact overwrite ------------------------------

@pytest.mark.parametrize("basis", ["signed_permutation", "hadamard"])
def test_orthonormal_overwrite(oracle_mod, basis):
    dk = dv = 64
    rng = np.random.default_rng(3)
    if basis == "signed_permutation":
        Kb = np.eye(dk)[rng.permutation(dk)] * rng.choice([-1.0, 1.0], (dk, 1))
    else:
        H = np.array([[1.0]])
        while H.shape[0] < dk:
            H = np.block([[H, H], [H, -H]])
        Kb = H[rng.permutation(dk)] / 8.0          # rows orthonormal, entries +-1/8 (bf16-exact)
    T = 48
    x = small(T=T, dk=dk, dv=dv, seed=4, h0_std=None)
    k = np.zeros((1, T, 1, dk), np.float32)
    k[0, :, 0] = Kb[:T]
    picks = [int(rng.integers(0, t + 1)) for t in range(T)]      # q_t = k_j for some j <= t
    qa = np.zeros_like(k)
    qa[0, :, 0] = Kb[picks]
    v = as_np(x.v).astype(np.float32)
    g = np.zeros((1, T, 1), np.float32)
    beta = np.ones((1, T, 1), np.float32)
    for f in (oracle_mod.gdn_recurrent, oracle_mod.gdn_chunked):
        o, hT = f(qa, k, v, g, beta, None)
        np.testing.assert_allclose(o[0, :, 0], v[0, picks, 0], rtol=0, atol=1e-12)
        S_ref = sum(np.outer(Kb[j], v[0, j, 0]) for j in range(T))
        np.testing.assert_allclose(hT[0, 0], S_ref, rtol=0, atol=1e-12)


# --- split / resume ---------------------------------------------------------------------

@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_split_resume_bitwise(oracle_mod, form):
    T, T1 = 200, 128
    x = small(B=2, T=T, Hv=2, dk=32, dv=64, seed=8)
    f = run1 if form == "recurrent" else run2
    kw = dict(state_qdq=True) if form == "recurrent" else dict(state_qdq=True, w_qdq=True)
    o, hT = f(oracle_mod, x, **kw)
    a = workloads.PrefillInputs(x.q[:, :T1], x.k[:, :T1], x.v[:, :T1], x.g[:, :T1], x.beta[:, :T1], x.h0, None)
    oa, ha = f(oracle_mod, a, **kw)
    fb = oracle_mod.gdn_recurrent if form == "recurrent" else oracle_mod.gdn_chunked
    ob, hb = fb(x.q[:, T1:], x.k[:, T1:], x.v[:, T1:], x.g[:, T1:], x.beta[:, T1:], ha, None, **kw)
    np.testing.assert_array_equal(np.concatenate([oa, ob], axis=1), o)
    np.testing.assert_array_equal(hb, hT)


# --- varlen == per-sequence runs; GQA == materialised repeat --------------------------------

def test_varlen_equals_dense(oracle_mod):
    lens = [0, 1, 63, 64, 65, 130]
    x = small(B=1, Hqk=1, Hv=2, dk=32, dv=64, seed=9, seqlens=lens)
    cu = x.cu_seqlens.tolist()
    for f in (run1, run2):
        o, hT = f(oracle_mod, x, state_qdq=True)
        for n, L in enumerate(lens):
            s = slice(cu[n], cu[n + 1])
            d = workloads.PrefillInputs(x.q[:, s], x.k[:, s], x.v[:, s], x.g[:, s], x.beta[:, s],
                                        x.h0[n:n + 1], None)
            od, hd = f(oracle_mod, d, state_qdq=True)
            np.testing.assert_array_equal(o[:, s], od)
            np.testing.assert_array_equal(hT[n], hd[0])
            if L == 0:
                np.testing.assert_array_equal(hT[n], as_np(x.h0)[n])


def test_gqa_equals_repeat(oracle_mod):
    x = small(B=2, T=100, Hqk=2, Hv=6, dk=16, dv=32, seed=10)
    G = 3
    r = workloads.PrefillInputs(x.q.repeat_interleave(G, dim=2), x.k.repeat_interleave(G, dim=2), x.v, x.g,
                                x.beta, x.h0, None)
    for f in (run1, run2):
        o, hT = f(oracle_mod, x, state_qdq=True)
        orr, hr = f(oracle_mod, r, state_qdq=True)
        np.testing.assert_array_equal(o, orr)
        np.testing.assert_array_equal(hT, hr)


# --- KDA with equal channels == GDN ---------------------------------------------------------

def test_kda_equal_channels_is_gdn(oracle_mod):
    x = small(B=1, T=150, Hv=2, dk=32, dv=64, seed=12)
    xk = workloads.PrefillInputs(x.q, x.k, x.v, x.g[..., None].expand(*x.g.shape, 32).contiguous(), x.beta,
                                 x.h0, None, kda=True)
    o1, h1 = run1(oracle_mod, x, state_qdq=True)
    o2, h2 = run2(oracle_mod, xk, state_qdq=True)
    assert rel(o2, o1) < 1e-12 and rel(h2, h1) < 1e-12


# --- decode == recurrence with a QDQ after every token --------------------------------------

@pytest.mark.parametrize("kda", [False, True])
def test_decode_equals_recurrence_period_one(oracle_mod, kda):
    d = workloads.decode(5, 3, 2, 16, 128, seed=13, kda=kda)
    o, st = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, kda=kda, state_qdq=True)
    tr = lambda t: t.transpose(0, 1).contiguous()   # the same tokens as N sequences of `steps`
    x = workloads.PrefillInputs(tr(d.q), tr(d.k), tr(d.v), tr(d.g), tr(d.beta), d.state, None, kda=kda)
    o1, h1 = run1(oracle_mod, x, state_qdq=True, qdq_period=1)
    np.testing.assert_array_equal(o, o1.transpose(1, 0, 2, 3))
    np.testing.assert_array_equal(st, h1)


# --- W QDQ ---------------------------------------------------------------------------------

@pytest.mark.parametrize("state_qdq", [False, True])
def test_w_qdq_closed_form(oracle_mod, state_qdq):
    """One chunk with g = 0 and beta = (1, 0, ..., 0): A = 0, so W has the single nonzero
    row k_0 and U the single row v_0. Then Delta_0 = v_0 - S0^T QDQ(k_0), Delta_r = 0 for r > 0,
    o_r = q_r^T S0 + (q_r . k_0) Delta_0 and S1 = S0 + k_0 Delta_0^T: a closed form that pins
    which operand W QDQ acts on and the tile it uses (all L x dk entries of W)."""
    T, dk, dv = 64, 32, 96
    x = small(T=T, dk=dk, dv=dv, seed=14)
    x.g.zero_()
    x.beta.zero_()
    x.beta[0, 0, 0] = 1.0
    q, k, v, S0 = as_np(x.q)[0, :, 0], as_np(x.k)[0, :, 0], as_np(x.v)[0, :, 0], as_np(x.h0)[0, 0]
    for w_qdq in (False, True):
        w0 = oracle_mod.tile_qdq_f64(k[0][None, :], dk)[0][0, 0] if w_qdq else k[0]
        d0 = v[0] - S0.T @ w0
        o_ref = q @ S0 + np.outer(q @ k[0], d0)
        S1 = S0 + np.outer(k[0], d0)
        if state_qdq:
            S1 = oracle_mod.tile_qdq_f64(S1, 64)[0][0]
        o, hT = run2(oracle_mod, x, w_qdq=w_qdq, state_qdq=state_qdq)
        assert rel(o[0, :, 0], o_ref) < 1e-12
        assert rel(hT[0, 0], S1) < 1e-12
    o1, h1 = run1(oracle_mod, x, state_qdq=state_qdq)   # W QDQ off: the recurrence agrees too
    o2, h2 = run2(oracle_mod, x, state_qdq=state_qdq)
    assert rel(o1, o2) < 1e-12 and rel(h1, h2) < 1e-12


def test_w_qdq_no_effect_from_zero_state(oracle_mod):
    """With S0 = 0 for a single chunk, W only meets a zero state: W QDQ cannot change anything."""
    x = small(T=64, dk=32, dv=64, seed=15, h0_std=None)
    a = run2(oracle_mod, x, w_qdq=False, state_qdq=True)
    b = run2(oracle_mod, x, w_qdq=True, state_qdq=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_w_qdq_changes_result_by_e4m3_size(oracle_mod):
    """Across many chunks W QDQ perturbs the output by roughly E4M3 relative precision
    (3 mantissa bits): visibly, but far below 1."""
    x = small(B=1, T=512, Hv=1, dk=64, dv=64, seed=16, h0_std=0.1)
    a, _ = run2(oracle_mod, x, w_qdq=False)
    b, _ = run2(oracle_mod, x, w_qdq=True)
    assert 1e-4 < rel(b, a) < 0.1


def test_empty_and_tiny_lengths(oracle_mod):
    """T = 0 leaves h0 untouched; T = 1 is a single recurrence step."""
    x = small(B=1, Hv=1, dk=16, dv=64, seed=17, seqlens=[0, 1, 0])
    o1, h1 = run1(oracle_mod, x, state_qdq=True)
    o2, h2 = run2(oracle_mod, x, state_qdq=True)
    h0 = as_np(x.h0)
    np.testing.assert_array_equal(h1[0], h0[0])
    np.testing.assert_array_equal(h1[2], h0[2])
    assert rel(h2, h1) < 1e-12 and rel(o2, o1) < 1e-12
