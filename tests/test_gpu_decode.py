"""gdn_decode_step on the GPU against the oracle's decode ("Torch GDN/KDA decode QAT with INT8
recurrent state", "Megatron-Core QAT/QAD workflow", step 3; "Add experimental GDN/KDA decode
and replay QAT": per-token FP8 state writes)."""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_OFF, TOL_QDQ, mask_for, rel, sample_units

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


def test_decode_full_size_sampled(gdn, oracle_mod):
    """512 sequences x 32 heads, dk = dv = 128, 64 steps with QDQ on every write; the oracle
    recomputes 48 sampled (sequence, head) units over all 64 steps."""
    d = workloads.workload("gdn_decode_n512_h32_d128_s64")
    o, st = run_gpu(gdn, d)
    units = sample_units(512, 32, 48, seed=3)
    oo, so = oracle_mod.gdn_decode(d.q, d.k, d.v, d.g, d.beta, d.state, state_qdq=True,
                                   unit_mask=mask_for(units, 512, 32))
    ns, hs = zip(*units)
    ns, hs = list(ns), list(hs)
    assert rel(o[:, ns, hs], oo[:, ns, hs]) <= TOL_QDQ
    assert rel(st[ns, hs], so[ns, hs]) <= TOL_QDQ
    for n, h in units:
        assert rel(st[n, h], so[n, h]) <= TOL_QDQ
    # the other units were updated too (not left at the initial state)
    assert not np.allclose(st[0, 0], d.state[0, 0].double().numpy())
