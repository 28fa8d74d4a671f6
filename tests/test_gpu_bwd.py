"""gdn_chunk_bwd / kda_chunk_bwd on the GPU against the fp64 gradient oracle.

The backward of the token recurrence with the state QDQ in the forward values and the identity in
the backward ("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core QAT/QAD
workflow" step 4; "GDN state/W QAT foundation": identity straight-through gradients). Bounds
(relative L2 per gradient tensor): 1e-3 with the state quantizer off; 2e-2 with it on (an fp32 and
an fp64 forward state can round to neighbouring codes at a boundary).
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_OFF, TOL_QDQ, rel, to_cuda

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def run(gdn, oracle_mod, x, state_qdq, codec="e4m3", with_dhT=True, seed=0):
    from oracle.grad import gdn_recurrent_grads
    gen = torch.Generator().manual_seed(seed)
    B, T = x.q.shape[:2]
    N, Hv, dk, dv = x.shape["N"], x.shape["Hv"], x.shape["dk"], x.shape["dv"]
    dout = torch.randn((B, T, Hv, dv), generator=gen)
    dhT = torch.randn((N, Hv, dk, dv), generator=gen) if with_dhT else None
    c = to_cuda(x)
    fn = gdn.kda_chunk_bwd if x.kda else gdn.gdn_chunk_bwd
    got = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, dout.cuda(),
             None if dhT is None else dhT.cuda(), state_qdq=state_qdq, codec=codec)
    torch.cuda.synchronize()
    ref = gdn_recurrent_grads(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, dout.double(),
                              None if dhT is None else dhT.double(), kda=x.kda, state_qdq=state_qdq, codec=codec)[:6]
    tol = TOL_QDQ if state_qdq else TOL_OFF
    for name, a, b in zip(NAMES, got, ref):
        if b.size == 0 or not np.any(b):
            continue
        e = rel(a.cpu().double().numpy(), b)
        assert e <= tol, (name, e)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 64), (64, 256)])
def test_bwd_shapes_no_qdq(gdn, oracle_mod, kda, dk, dv):
    x = workloads.prefill(1, 0, 2, 4, dk, dv, seed=80 + dk + dv + kda, kda=kda, h0_std=0.1, seqlens=[0, 1, 63, 64, 130])
    run(gdn, oracle_mod, x, False, seed=1)


@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("codec", ["e4m3", "int8"])
def test_bwd_state_qdq(gdn, oracle_mod, kda, codec):
    x = workloads.prefill(1, 0, 1, 2, 128, 128, seed=90 + kda, kda=kda, h0_std=0.1, seqlens=[64, 150, 20])
    run(gdn, oracle_mod, x, True, codec=codec, seed=2)


@pytest.mark.parametrize("kda", [False, True])
def test_bwd_more_units_than_ctas(gdn, oracle_mod, kda):
    """160 (sequence, head, slab) units on a grid of at most one CTA per SM: some CTAs walk a
    second unit (persistent loop), with ragged lengths and state QDQ on."""
    lens = torch.randint(1, 90, (40,), generator=torch.Generator().manual_seed(97)).tolist()
    x = workloads.prefill(1, 0, 2, 4, 64, 64, seed=98 + kda, kda=kda, h0_std=0.1, seqlens=lens)
    run(gdn, oracle_mod, x, True, seed=4)


def test_bwd_dense_no_final_grad(gdn, oracle_mod):
    x = workloads.prefill(2, 96, 2, 2, 128, 128, seed=95, h0_std=0.1)
    run(gdn, oracle_mod, x, True, with_dhT=False, seed=3)


def test_bwd_refuses_w_qdq(gdn):
    x = workloads.prefill(1, 64, 1, 1, 64, 64, seed=96)
    c = to_cuda(x)
    a, _, _ = gdn.gdnqat._chunk_args(c["q"], c["k"], c["v"], c["g"], c["beta"], None, None, True, True, 1.0,
                                     torch.empty(0, device="cuda"), None, False)
    assert gdn.load().gdn_chunk_bwd_workspace_size(__import__("ctypes").byref(a)) == 0


def test_bwd_full_size_sampled(gdn, oracle_mod):
    """The benchmarked backward workload (B4 H16 T4096 d128, state QDQ straight through) in the
    launch configuration bench.py times; the oracle recomputes one sampled (sequence, head) unit
    over all 4096 tokens (fp64 autograd, ~2 minutes; no GQA: the unit's dq and dk are its own)."""
    from oracle.grad import gdn_recurrent_grads
    x = workloads.workload("gdn_bwd_b4_h16_t4096_d128")
    gen = torch.Generator().manual_seed(12)
    dout = torch.randn((4, 4096, 16, 128), generator=gen)
    c = to_cuda(x)
    got = gdn.gdn_chunk_bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], None, dout.cuda(), state_qdq=True)
    torch.cuda.synchronize()
    units = [(3, 12)]
    ref = gdn_recurrent_grads(x.q, x.k, x.v, x.g, x.beta, x.h0, None, dout.double(), None, state_qdq=True,
                              units=units)[:6]
    got = [t.cpu().double().numpy() for t in got]
    for n, h in units:
        sel = {"dq": (n, slice(None), h), "dk": (n, slice(None), h), "dv": (n, slice(None), h),
               "dg": (n, slice(None), h), "dbeta": (n, slice(None), h), "dh0": (n, h)}
        for name, a, b in zip(NAMES, got, ref):
            e = rel(a[sel[name]], b[sel[name]])
            assert e <= TOL_QDQ, (name, n, h, e)


def test_kda_bwd_full_size_consistency(gdn, oracle_mod):
    """The KDA backward workload (B2 H32 T8192 d128, state QDQ straight through) in the launch
    configuration bench.py times. A unit's gradients depend only on its own sequence and head
    (no GQA here) and the kernels sum in a fixed order, so sequence 1's gradients must equal, bit
    for bit, those of the same call on sequence 1 alone. Its first 512 tokens, run alone, are
    checked against the oracle for one (sequence, head) unit."""
    from oracle.grad import gdn_recurrent_grads
    x = workloads.workload("kda_bwd_b2_h32_t8192_d128")
    gen = torch.Generator().manual_seed(13)
    dout = torch.randn((2, 8192, 32, 128), generator=gen)
    c = to_cuda(x)
    full = gdn.kda_chunk_bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], None, dout.cuda(), state_qdq=True)
    one = lambda t: t[1:2].contiguous()
    alone = gdn.kda_chunk_bwd(one(c["q"]), one(c["k"]), one(c["v"]), one(c["g"]), one(c["beta"]), one(c["h0"]), None,
                              dout[1:2].contiguous().cuda(), state_qdq=True)
    torch.cuda.synchronize()
    for name, a, b in zip(NAMES, full, alone):
        assert torch.equal(a[1:2], b), name
    T = 512
    pre = lambda t: t[1:2, :T].contiguous()
    got = gdn.kda_chunk_bwd(pre(c["q"]), pre(c["k"]), pre(c["v"]), pre(c["g"]), pre(c["beta"]), one(c["h0"]), None,
                            dout[1:2, :T].contiguous().cuda(), state_qdq=True)
    torch.cuda.synchronize()
    h = 21
    ref = gdn_recurrent_grads(x.q[1:2, :T], x.k[1:2, :T], x.v[1:2, :T], x.g[1:2, :T], x.beta[1:2, :T], x.h0[1:2],
                              None, dout[1:2, :T].double(), None, kda=True, state_qdq=True, units=[(0, h)])[:6]
    got = [t.cpu().double().numpy() for t in got]
    sel = {"dq": (0, slice(None), h), "dk": (0, slice(None), h), "dv": (0, slice(None), h),
           "dg": (0, slice(None), h), "dbeta": (0, slice(None), h), "dh0": (0, h)}
    for name, a, b in zip(NAMES, got, ref):
        e = rel(a[sel[name]], b[sel[name]])
        assert e <= TOL_QDQ, (name, e)
