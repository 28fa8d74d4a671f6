"""The INT8 block state codec on the GPU against the fp64 oracle.

Codec (summary of "Torch GDN/KDA decode QAT with INT8 recurrent state"; signed INT8 codes,
a scale per 32-value block): one scale per key row and 32 value columns, amax / 127 with the zero
guard, codes = nearest integer (ties to even) within +-127. The standalone op is compared bit for
bit with the oracle's fp32 definition; the fused uses (chunk carry, decode, handoff) within the
QDQ bound (rel-L2 <= 2e-2), plus teacher-forced decode steps that take the same decisions.
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_QDQ, bits, compare_units, rel, to_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,block", [(1, 32, 32), (64, 128, 32), (33, 70, 32), (5, 1000, 128), (7, 45, 7),
                                             (3, 17, 1), (16384 * 2, 128, 32)])
def test_standalone_bit_exact(gdn, oracle_mod, rows, cols, block):
    gen = torch.Generator().manual_seed(rows * 1000 + cols)
    x = torch.randn((rows, cols), generator=gen) * torch.exp(torch.randn((rows, 1), generator=gen) * 4)
    x[0, : min(cols, 5)] = 0.0
    if rows > 2:
        x[1] = 0.0                                   # an all-zero row: scale 1, zeros out
        x[2] *= 1e-39                                # subnormal scales: the IEEE-divide path
    y_ref, s_ref = oracle_mod.int8_block_qdq_f32(x.numpy(), block)
    y, s = gdn.int8_block_qdq(x.cuda(), block)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y), bits(y_ref))
    np.testing.assert_array_equal(bits(s), bits(s_ref))
    xi = x.cuda()
    gdn.int8_block_qdq(xi, block, y=xi, scales=False)   # in place
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(xi), bits(y_ref))


def run_chunk(gdn, x, w_qdq, path):
    c = to_cuda(x)
    fn = gdn.kda_chunk_fwd if x.kda else gdn.gdn_chunk_fwd
    ws = torch.empty(256, dtype=torch.uint8, device="cuda") if path == "fused" else None
    o, hT = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, state_qdq=True, w_qdq=w_qdq,
               workspace=ws, codec="int8")
    torch.cuda.synchronize()
    return o, hT


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (128, 64), (64, 64), (64, 256)])
@pytest.mark.parametrize("w_qdq", [False, True])
def test_chunk_int8_state(gdn, oracle_mod, kda, path, dk, dv, w_qdq):
    """Varlen with tails and exact multiples of 64, GQA; dk = 128 through the tensor-core split or
    (minimum workspace) the fused / CUDA-core kernel, dk = 64 on CUDA cores."""
    if dk == 64 and path == "fused":
        pytest.skip("dk = 64 has a single path")
    x = workloads.prefill(1, 0, 2, 4, dk, dv, seed=41 + dk + dv, kda=kda, h0_std=0.1, seqlens=[1, 64, 100, 192, 130])
    o, hT = run_chunk(gdn, x, w_qdq, path)
    f = oracle_mod.gdn_chunked if w_qdq else oracle_mod.gdn_recurrent
    kw = dict(w_qdq=True) if w_qdq else {}
    oref, href = f(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=True, codec="int8", **kw)
    units = [(n, h) for n in range(5) for h in range(4)]
    compare_units(x, units, o, hT, oref, href, TOL_QDQ)
    # the codec matters: E4M3 state QDQ gives a different final state
    oe, he = f(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=kda, state_qdq=True, **kw)
    assert rel(hT.cpu().double().numpy(), he) > 5 * rel(hT.cpu().double().numpy(), href)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 256), (128, 64)])
def test_decode_int8(gdn, oracle_mod, kda, dk, dv):
    d = workloads.decode(6, 5, 4, dk, dv, seed=50 + dk + dv + kda, kda=kda, state_std=0.05)
    st = d.state.cuda()
    outs = []
    for s in range(6):
        outs.append(gdn.gdn_decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.g[s].cuda(), d.beta[s].cuda(),
                                        st, kda=kda, codec="int8"))
    torch.cuda.synchronize()
    o = torch.stack(outs).cpu().double().numpy()
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, kda=kda, state_qdq=True, codec="int8")
    assert rel(o, oo) <= TOL_QDQ and rel(st.cpu().double().numpy(), so) <= TOL_QDQ


def test_decode_int8_teacher_forced(gdn, oracle_mod):
    """Each step starts the oracle from the GPU's stored state: nearly every element is then the
    same integer times the same scale."""
    d = workloads.decode(8, 64, 8, 128, 128, seed=60, state_std=0.05)
    st = d.state.cuda()
    for s in range(8):
        before = st.cpu()
        o = gdn.gdn_decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.g[s].cuda(), d.beta[s].cuda(), st,
                                codec="int8")
        torch.cuda.synchronize()
        oo, so = oracle_mod.gdn_decode(d.q[s:s + 1], d.k[s:s + 1], d.v[s:s + 1], d.g[s:s + 1], d.beta[s:s + 1],
                                       before, state_qdq=True, codec="int8")
        g_st = st.cpu().double().numpy()
        assert rel(o.cpu().double().numpy(), oo[0]) <= 1e-5
        same = np.isclose(g_st, so, rtol=1e-5, atol=0).mean()
        assert same >= 0.999, same


@pytest.mark.parametrize("kda", [False, True])
def test_handoff_int8_teacher_forced(gdn, oracle_mod, kda):
    """The handoff with the INT8 codec: every decode token teacher forced against the oracle's
    decode step (handoff QDQ first), o within 1e-5 and >= 99.9 % identical stored elements."""
    L, P = 90, 40
    x = workloads.prefill(1, L, 2, 2, 128, 128, seed=61, kda=kda, h0_std=0.1)
    c = to_cuda(x)
    fn = gdn.kda_prefill_decode_fwd if kda else gdn.gdn_prefill_decode_fwd

    def gpu_upto(t):
        cut = lambda v: v[:, :t].contiguous()
        o, hT = fn(cut(c["q"]), cut(c["k"]), cut(c["v"]), cut(c["g"]), cut(c["beta"]), c["h0"], None, [P],
                   state_qdq=True, w_qdq=True, codec="int8")
        torch.cuda.synchronize()
        return o.cpu().double().numpy(), hT.cpu().double().numpy()

    _, S = gpu_upto(P)
    for t in range(P, L):
        o_next, S_next = gpu_upto(t + 1)
        start = S if t > P else oracle_mod.int8_block_qdq_f64(S, 32)[0]
        step = lambda v: v[:, t:t + 1].transpose(0, 1).contiguous()
        oo, so = oracle_mod.gdn_decode(step(x.q), step(x.k), step(x.v), step(x.g), step(x.beta), start, kda=kda,
                                       state_qdq=True, codec="int8")
        assert rel(o_next[0, t], oo[0, 0]) <= 1e-5, t
        same = np.isclose(S_next, so, rtol=1e-5, atol=0).mean()
        assert same >= 0.999, (t, same)
        S = S_next


def test_standalone_full_workload_bit_exact(gdn, oracle_mod):
    """The benchmarked INT8 block QDQ workload (16384 x [128 x 128] fp32, 32-column blocks), in
    the launch configuration bench.py times, bit for bit against the oracle's fp32 definition."""
    d = workloads.workload("int8_state_n512_h32_d128")
    x = d.x.reshape(-1, 128)
    y_ref, s_ref = oracle_mod.int8_block_qdq_f32(x.numpy(), 32)
    y, s = gdn.int8_block_qdq(x.cuda(), 32)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), bits(y_ref)) and np.array_equal(bits(s), bits(s_ref))


def test_decode_int8_full_size_sampled(gdn, oracle_mod):
    """The benchmarked INT8 decode workload (512 sequences x 32 heads, 64 steps, INT8 block QDQ
    on every write); the oracle recomputes 48 sampled (sequence, head) units over all 64 steps."""
    from helpers import UNIT_SANITY_PER_TOKEN, mask_for, sample_units
    d = workloads.workload("gdn_decode_int8_n512_h32_d128_s64")
    st = d.state.cuda()
    outs = []
    for s in range(64):
        outs.append(gdn.gdn_decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.g[s].cuda(), d.beta[s].cuda(),
                                        st, codec="int8"))
    torch.cuda.synchronize()
    o = torch.stack(outs).cpu().double().numpy()
    st = st.cpu().double().numpy()
    units = sample_units(512, 32, 48, seed=3)
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, state_qdq=True, codec="int8",
                                   unit_mask=mask_for(units, 512, 32))
    ns, hs = (list(t) for t in zip(*units))
    assert rel(o[:, ns, hs], oo[:, ns, hs]) <= TOL_QDQ
    assert rel(st[ns, hs], so[ns, hs]) <= TOL_QDQ
    for n, h in units:
        assert rel(st[n, h], so[n, h]) <= UNIT_SANITY_PER_TOKEN
