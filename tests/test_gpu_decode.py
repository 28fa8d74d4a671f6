"""gdn_decode_step on the GPU against the oracle's decode ("Torch GDN/KDA decode QAT with INT8
recurrent state", "Megatron-Core QAT/QAD workflow", step 3; "Add experimental GDN/KDA decode
and replay QAT": per-token FP8 state writes)."""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_QDQ, UNIT_SANITY_PER_TOKEN, mask_for, rel, sample_units

pytestmark = pytest.mark.gpu


def run_gpu(gdn, d, steps=None, state_qdq=True):
    steps = d.q.shape[0] if steps is None else steps
    st = d.state.cuda()
    outs = []
    for s in range(steps):
        o = gdn.gdn_decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.g[s].cuda(), d.beta[s].cuda(), st,
                                state_qdq=state_qdq, kda=d.kda)
        outs.append(o)
    torch.cuda.synchronize()
    return torch.stack(outs).cpu().double().numpy(), st.cpu().double().numpy()


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq", [False, True])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 256), (128, 64)])
def test_decode_small(gdn, oracle_mod, kda, state_qdq, dk, dv):
    d = workloads.decode(6, 5, 4, dk, dv, seed=dk + dv + kda, kda=kda, state_std=0.05)
    o, st = run_gpu(gdn, d, state_qdq=state_qdq)
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, kda=kda, state_qdq=state_qdq)
    tol = TOL_QDQ if state_qdq else 1e-5     # fp32 CUDA-core arithmetic: far inside 1e-3 without QDQ
    assert rel(o, oo) <= tol and rel(st, so) <= tol, (rel(o, oo), rel(st, so))


def test_decode_gqa(gdn, oracle_mod):
    d = workloads.decode(4, 3, 4, 128, 128, seed=9)
    # 2 q/k heads shared by 4 value heads: keep the first 2 q/k heads
    d.q = d.q[:, :, :2].contiguous()
    d.k = d.k[:, :, :2].contiguous()
    o, st = run_gpu(gdn, d)
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, state_qdq=True)
    assert rel(o, oo) <= TOL_QDQ and rel(st, so) <= TOL_QDQ


@pytest.fixture(scope="module")
def full_decode():
    return workloads.workload("gdn_decode_n512_h32_d128_s64")


@pytest.mark.parametrize("state_qdq", [True, False])
def test_decode_full_size_sampled(gdn, oracle_mod, full_decode, state_qdq):
    """512 sequences x 32 heads, dk = dv = 128, 64 steps (QDQ on every write, or off); the
    oracle recomputes 48 sampled (sequence, head) units over all 64 steps. rel-L2 is taken
    over all sampled units together."""
    d = full_decode
    o, st = run_gpu(gdn, d, state_qdq=state_qdq)
    units = sample_units(512, 32, 48, seed=3)
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, state_qdq=state_qdq,
                                   unit_mask=mask_for(units, 512, 32))
    ns, hs = (list(t) for t in zip(*units))
    tol = TOL_QDQ if state_qdq else 1e-5
    assert rel(o[:, ns, hs], oo[:, ns, hs]) <= tol
    assert rel(st[ns, hs], so[ns, hs]) <= tol
    for n, h in units:
        assert rel(st[n, h], so[n, h]) <= (UNIT_SANITY_PER_TOKEN if state_qdq else tol)
    assert not np.allclose(st[0, 0], d.state[0, 0].double().numpy())   # every unit was updated


def test_decode_teacher_forced_steps(gdn, oracle_mod, full_decode):
    """Each of the first 8 steps starts the oracle from the GPU's own stored state, so both
    sides take the QDQ decisions on (nearly) the same inputs: the per-step result is then
    close to exact, not just within the end-to-end bound."""
    d = full_decode
    units = sample_units(512, 32, 32, seed=5)
    m = mask_for(units, 512, 32)
    ns, hs = (list(t) for t in zip(*units))
    st = d.state.cuda()
    for s in range(8):
        before = st.cpu()
        o = gdn.gdn_decode_step(d.q[s].cuda(), d.k[s].cuda(), d.v[s].cuda(), d.g[s].cuda(), d.beta[s].cuda(), st)
        torch.cuda.synchronize()
        oo, so = oracle_mod.gdn_decode(d.q[s:s + 1], d.k[s:s + 1], d.v[s:s + 1], d.g[s:s + 1], d.beta[s:s + 1],
                                       before, state_qdq=True, unit_mask=m)
        g_st = st.cpu().double().numpy()
        assert rel(o.cpu().double().numpy()[ns, hs], oo[0][ns, hs]) <= 1e-5
        assert rel(g_st[ns, hs], so[ns, hs]) <= 2e-3
        # nearly every stored element is the same E4M3 value times the same scale
        same = np.isclose(g_st[ns, hs], so[ns, hs], rtol=1e-5, atol=0).mean()
        assert same >= 0.999, same
