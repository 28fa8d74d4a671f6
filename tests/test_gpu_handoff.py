"""gdn_prefill_decode_fwd / kda_prefill_decode_fwd on the GPU against the fp64 oracle.

Schedule ("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD
workflow", steps 2-3): per sequence the first prefill_lengths[n] tokens run as chunked prefill
without internal state QDQ, the state is QDQ'd at the handoff when tokens remain, and every
remaining token is a teacher-forced decode step that QDQs the state before storing it.
Bounds: rel-L2 <= 1e-3 with QDQ off, <= 2e-2 with QDQ on (as for the chunked forward).
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_OFF, TOL_QDQ, compare_units, rel, to_cuda

pytestmark = pytest.mark.gpu


def run_gpu(gdn, x, P, state_qdq, w_qdq, hT_alias=False):
    c = to_cuda(x)
    fn = gdn.kda_prefill_decode_fwd if x.kda else gdn.gdn_prefill_decode_fwd
    hT = c["h0"] if (hT_alias and c["h0"] is not None) else None
    o, hT = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, P, state_qdq=state_qdq,
               w_qdq=w_qdq, hT=hT)
    torch.cuda.synchronize()
    return o, hT


def check(gdn, oracle_mod, x, P, state_qdq, w_qdq, hT_alias=False):
    """o and hT against the oracle. With state QDQ every decode token QDQs the state; an fp32
    and an fp64 state a few ulps apart then round some element to neighbouring E4M3 values,
    and from there on the two trajectories carry independent quantization noise (a few
    percent of the affected units' values). hT is therefore bounded here only where no
    decode token ran (whole-sequence prefixes, no state QDQ inside the prefill); the decode
    tokens' state is checked step by step in test_teacher_forced_decode_tokens."""
    o, hT = run_gpu(gdn, x, P, state_qdq, w_qdq, hT_alias)
    oref, href = oracle_mod.gdn_prefill_decode(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, P, kda=x.kda,
                                               state_qdq=state_qdq, w_qdq=w_qdq)
    N, Hv = x.shape["N"], x.shape["Hv"]
    tol = TOL_QDQ if (state_qdq or w_qdq) else TOL_OFF
    if not state_qdq:
        return compare_units(x, [(n, h) for n in range(N) for h in range(Hv)], o, hT, oref, href, tol)
    o_g, h_g = o.cpu().double().numpy(), hT.cpu().double().numpy()
    assert rel(o_g, oref) <= tol, rel(o_g, oref)
    B, T = x.q.shape[:2]
    lens = x.cu_seqlens.diff().tolist() if x.cu_seqlens is not None else [T] * B
    whole = [n for n in range(N) if P[n] == lens[n]]
    if whole:
        assert rel(h_g[whole], href[whole]) <= (TOL_OFF if not w_qdq else TOL_QDQ)


LENS = [0, 1, 64, 100, 128, 130, 200, 333]
PRE = [0, 0, 64, 37, 64, 130, 150, 290]
MODES = [(False, False), (True, False), (False, True), (True, True)]


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 256)])
@pytest.mark.parametrize("state_qdq,w_qdq", MODES)
def test_varlen_prefix_mix(gdn, oracle_mod, kda, dk, dv, state_qdq, w_qdq):
    """Empty sequences, empty prefixes, whole-sequence prefixes, prefixes on and off the
    64-token grid, GQA (2 q/k heads for 4 v-heads); dk = 128 takes the tensor-core prefill."""
    x = workloads.prefill(1, 0, 2, 4, dk, dv, seed=31, kda=kda, h0_std=0.1, seqlens=LENS, state_qdq=state_qdq,
                          w_qdq=w_qdq)
    check(gdn, oracle_mod, x, PRE, state_qdq, w_qdq)


@pytest.mark.parametrize("kda", [False, True])
def test_dense_batch_and_alias(gdn, oracle_mod, kda):
    """The pages' example shape: 128-token sequences, 64-token prefill; hT written over h0."""
    x = workloads.prefill(3, 128, 2, 4, 128, 128, seed=32, kda=kda, h0_std=0.1, state_qdq=True, w_qdq=True)
    check(gdn, oracle_mod, x, [64, 64, 64], True, True, hT_alias=True)
    check(gdn, oracle_mod, x, [0, 128, 17], True, True)


@pytest.mark.parametrize("kda", [False, True])
def test_whole_prefix_matches_chunk_forward_bitwise(gdn, kda):
    """prefill_lengths = L: the handoff is the chunked prefill with state QDQ off, bit for bit
    (the same kernels run the same tokens)."""
    x = workloads.prefill(1, 0, 2, 4, 128, 128, seed=33, kda=kda, h0_std=0.1, seqlens=[5, 64, 130, 200])
    c = to_cuda(x)
    fwd = gdn.kda_chunk_fwd if kda else gdn.gdn_chunk_fwd
    o1, h1 = fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, state_qdq=False, w_qdq=True)
    o2, h2 = run_gpu(gdn, x, [5, 64, 130, 200], True, True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("kda", [False, True])
def test_no_prefix_matches_decode_steps(gdn, kda):
    """prefill_lengths = 0 and state QDQ: QDQ(h0), then every token a decode step (150 of
    them). Against the library's own tile QDQ and decode step: the same state codes except
    where the fused QDQ's reciprocal and the standalone op's IEEE divide land on opposite
    sides of a rounding boundary (a few in 10^6 elements)."""
    T, N, H = 150, 3, 4
    x = workloads.prefill(N, T, 2, H, 128, 128, seed=34, kda=kda, h0_std=0.1, state_qdq=True)
    c = to_cuda(x)
    o, hT = run_gpu(gdn, x, [0] * N, True, False)
    st, _ = gdn.fp8_tile_qdq(c["h0"].reshape(N * H, 128, 128), 64)
    st = st.reshape(N, H, 128, 128).contiguous()
    od = []
    for t in range(T):
        od.append(gdn.gdn_decode_step(c["q"][:, t].contiguous(), c["k"][:, t].contiguous(), c["v"][:, t].contiguous(),
                                      c["g"][:, t].contiguous(), c["beta"][:, t].contiguous(), st, state_qdq=True,
                                      kda=kda))
    od = torch.stack(od, dim=1)
    same = (hT == st).float().mean().item()
    assert same >= 0.999, same
    rel = ((o - od).norm() / od.norm()).item()
    assert rel < 1e-3, rel


def test_rejects_bad_lengths(gdn):
    x = workloads.prefill(2, 64, 1, 2, 128, 128, seed=35)
    with pytest.raises(gdn.GdnError):
        run_gpu(gdn, x, [65, 0], True, False)
    with pytest.raises(ValueError):
        run_gpu(gdn, x, [1, 2, 3], True, False)


@pytest.mark.parametrize("kda,dv", [(False, 128), (False, 64), (True, 128), (True, 64)])
def test_teacher_forced_decode_tokens(gdn, oracle_mod, kda, dv):
    """Every decode token of the handoff, teacher forced: the GPU's state after t tokens (the
    same call on the sequence cut after token t; the kernels are deterministic) is fed to the
    oracle's decode step for token t (preceded by the handoff QDQ when t is the first decode
    token), and the result is compared with the GPU's state after t + 1 tokens. Both sides
    then take each QDQ decision on nearly the same input, as in the decode step's own
    teacher-forced test: o of the token within 1e-5, and >= 99.9 % of the stored state the
    same E4M3 value times the same scale. The handoff QDQ (before the first decode token's o)
    divides exactly on the GPU and is compared with the oracle's fp32 QDQ, so the same codes
    result; the per-token QDQs after each o use the rounded reciprocal of the scale."""
    L, P = 100, 37
    x = workloads.prefill(1, L, 2, 2, 128, dv, seed=36, kda=kda, h0_std=0.1, state_qdq=True, w_qdq=True)
    c = to_cuda(x)
    fn = gdn.kda_prefill_decode_fwd if kda else gdn.gdn_prefill_decode_fwd

    def gpu_upto(t):   # (o, hT) of the handoff on the first t tokens
        cut = lambda v: v[:, :t].contiguous()
        o, hT = fn(cut(c["q"]), cut(c["k"]), cut(c["v"]), cut(c["g"]), cut(c["beta"]), c["h0"], None, [P],
                   state_qdq=True, w_qdq=True)
        torch.cuda.synchronize()
        return o.cpu().double().numpy(), hT.cpu().double().numpy()

    _, S = gpu_upto(P)
    for t in range(P, L):
        o_next, S_next = gpu_upto(t + 1)
        start = S
        if t == P:   # the handoff QDQ: in fp32 with the IEEE quotient, as the GPU takes it
            start = oracle_mod.tile_qdq_f32(S.astype(np.float32).reshape(-1, 128, dv), 64)[0].reshape(S.shape)
        step = lambda v: v[:, t:t + 1].transpose(0, 1).contiguous()   # token t as one decode step, N = 1
        oo, so = oracle_mod.gdn_decode(step(x.q), step(x.k), step(x.v), step(x.g), step(x.beta), start, kda=kda,
                                       state_qdq=True)
        assert rel(o_next[0, t], oo[0, 0]) <= 1e-5, (t, rel(o_next[0, t], oo[0, 0]))
        assert rel(S_next, so) <= 2e-3, (t, rel(S_next, so))
        same = np.isclose(S_next, so, rtol=1e-5, atol=0).mean()
        assert same >= 0.999, (t, same)
        S = S_next


def test_handoff_full_size_sampled(gdn, oracle_mod):
    """The benchmarked handoff workload (256 sequences x 128 tokens, 64-token prefix, H16 d128,
    state + W QDQ) in the launch configuration bench.py times; the oracle recomputes 32 sampled
    (sequence, head) units: o within the QDQ bound over the sampled units together, the final
    states free of gross errors (their decode tokens carry independent quantization noise, see
    check()), and every decode token's step checked teacher forced in
    test_teacher_forced_decode_tokens."""
    from helpers import UNIT_SANITY_PER_TOKEN, mask_for, sample_units
    x = workloads.workload("handoff_n256_t128_p64_h16_d128")
    c = to_cuda(x)
    o, hT = gdn.gdn_prefill_decode_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], None, x.prefill_lengths,
                                       state_qdq=True, w_qdq=True)
    torch.cuda.synchronize()
    units = sample_units(256, 16, 32, seed=7)
    oref, href = oracle_mod.gdn_prefill_decode(x.q, x.k, x.v, x.g, x.beta, x.h0, None, x.prefill_lengths,
                                               state_qdq=True, w_qdq=True, unit_mask=mask_for(units, 256, 16))
    o, hT = o.cpu().double().numpy(), hT.cpu().double().numpy()
    ns, hs = (list(t) for t in zip(*units))
    assert rel(o[ns, :, hs], oref[ns, :, hs]) <= TOL_QDQ
    for n, h in units:
        assert rel(hT[n, h], href[n, h]) <= UNIT_SANITY_PER_TOKEN
        assert rel(o[n, :64, h], oref[n, :64, h]) <= TOL_QDQ   # the prefix: W QDQ, no state QDQ
