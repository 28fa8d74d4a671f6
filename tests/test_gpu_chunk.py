"""gdn_chunk_fwd / kda_chunk_fwd on the GPU against the fp64 oracle.

State QDQ at every 64th token of a sequence with one scale per full-key x 64-value-column
tile; W QDQ with one scale per (sequence, head, chunk) ("GDN state/W QAT foundation", "What
does this PR do?"); KDA per-key-channel decay ("Add KDA prefill numerical emulation for QAT").
With W QDQ off the oracle is the token-by-token recurrence, with W QDQ on the chunked form
(W QDQ exists only there). Bounds: rel-L2 <= 1e-3 with QDQ off, <= 2e-2 with QDQ on.
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import TOL_OFF, TOL_QDQ, compare_units, mask_for, sample_units, to_cuda

pytestmark = pytest.mark.gpu


# dk = 128 has two paths: "split" (the workspace holds the per-chunk staging: a parallel prep
# kernel, then the state chain, both on tensor cores) and "fused" (the minimum 256-byte
# workspace: one kernel; for KDA the CUDA-core kernel)
PATHS = ["split", "fused"]


def run_gpu(gdn, x, state_qdq, w_qdq, hT_alias=False, path="split"):
    c = to_cuda(x)
    fn = gdn.kda_chunk_fwd if x.kda else gdn.gdn_chunk_fwd
    hT = c["h0"] if (hT_alias and c["h0"] is not None) else None
    ws = torch.empty(256, dtype=torch.uint8, device="cuda") if path == "fused" else None
    o, hT = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, state_qdq=state_qdq,
               w_qdq=w_qdq, hT=hT, workspace=ws)
    torch.cuda.synchronize()
    return o, hT


def run_oracle(oracle_mod, x, state_qdq, w_qdq, units=None):
    N, Hv = x.shape["N"], x.shape["Hv"]
    m = None if units is None else mask_for(units, N, Hv)
    if w_qdq:
        return oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=x.kda,
                                      state_qdq=state_qdq, w_qdq=True, unit_mask=m)
    return oracle_mod.gdn_recurrent(x.q, x.k, x.v, x.g, x.beta, x.h0, x.cu_seqlens, kda=x.kda,
                                    state_qdq=state_qdq, unit_mask=m)


def check(gdn, oracle_mod, x, state_qdq, w_qdq, units=None, hT_alias=False, path="split"):
    o, hT = run_gpu(gdn, x, state_qdq, w_qdq, hT_alias, path)
    oref, href = run_oracle(oracle_mod, x, state_qdq, w_qdq, units)
    if units is None:
        units = [(n, h) for n in range(x.shape["N"]) for h in range(x.shape["Hv"])]
    tol = TOL_QDQ if (state_qdq or w_qdq) else TOL_OFF
    return compare_units(x, units, o, hT, oref, href, tol)


QDQ_MODES = [(False, False), (True, False), (False, True), (True, True)]


@pytest.mark.parametrize("state_qdq,w_qdq", QDQ_MODES)
def test_small_workload(gdn, oracle_mod, state_qdq, w_qdq):
    """B1 H2 T256 d64 (4 chunks of 64), h0 = 0, the small parity workload."""
    x = workloads.workload("gdn_b1_h2_t256_d64")
    check(gdn, oracle_mod, x, state_qdq, w_qdq)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 200])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 256), (128, 64), (128, 256)])
def test_lengths_and_shapes(gdn, oracle_mod, T, dk, dv, path):
    if dk == 64 and path == "fused":
        pytest.skip("dk = 64 has a single path")
    x = workloads.prefill(2, T, 1, 2, dk, dv, seed=T + dk + dv, h0_std=0.1)
    check(gdn, oracle_mod, x, True, False, path=path)
    check(gdn, oracle_mod, x, False, False, path=path)
    if dk == 128:
        check(gdn, oracle_mod, x, True, True, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("state_qdq,w_qdq", QDQ_MODES)
def test_varlen_gqa(gdn, oracle_mod, kda, state_qdq, w_qdq, path):
    lens = [0, 1, 63, 64, 65, 129, 300]
    x = workloads.prefill(1, 0, 2, 4, 128, 128, seed=31 + kda, h0_std=0.1, seqlens=lens, kda=kda)
    check(gdn, oracle_mod, x, state_qdq, w_qdq, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_final_state_aliases_h0(gdn, oracle_mod, path):
    x = workloads.prefill(2, 150, 2, 2, 128, 128, seed=41, h0_std=0.1)
    check(gdn, oracle_mod, x, True, True, hT_alias=True, path=path)


def test_paths_agree_closely(gdn):
    """The two dk = 128 paths compute the same arithmetic (operands split the same way, the same
    QDQ epilogues); on a QDQ-off case their outputs agree far inside the oracle bound."""
    x = workloads.prefill(2, 333, 2, 4, 128, 128, seed=44, h0_std=0.1)
    o1, h1 = run_gpu(gdn, x, False, False, path="split")
    o2, h2 = run_gpu(gdn, x, False, False, path="fused")
    from helpers import rel
    assert rel(o1.cpu().double().numpy(), o2.cpu().double().numpy()) <= 1e-5
    assert rel(h1.cpu().double().numpy(), h2.cpu().double().numpy()) <= 1e-5


def test_zero_initial_state_and_no_final_state(gdn, oracle_mod):
    x = workloads.prefill(1, 100, 1, 1, 64, 64, seed=42, h0_std=None)
    c = to_cuda(x)
    o, hT = gdn.gdn_chunk_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], None, None, state_qdq=True,
                              output_final_state=False)
    assert hT is None
    oref, _ = run_oracle(oracle_mod, x, True, False)
    torch.cuda.synchronize()
    from helpers import rel
    assert rel(o.cpu().double().numpy(), oref) <= TOL_QDQ


@pytest.mark.parametrize("path", PATHS)
def test_kda_small(gdn, oracle_mod, path):
    x = workloads.prefill(2, 200, 2, 2, 128, 128, seed=43, kda=True, h0_std=0.1)
    check(gdn, oracle_mod, x, False, False, path=path)
    check(gdn, oracle_mod, x, True, True, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 200])
@pytest.mark.parametrize("dv", [64, 128, 256])
def test_kda_lengths_and_shapes(gdn, oracle_mod, T, dv, path):
    x = workloads.prefill(2, T, 1, 2, 128, dv, seed=7 * T + dv, h0_std=0.1, kda=True)
    check(gdn, oracle_mod, x, True, False, path=path)
    check(gdn, oracle_mod, x, False, False, path=path)
    check(gdn, oracle_mod, x, True, True, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_kda_final_state_aliases_h0(gdn, oracle_mod, path):
    x = workloads.prefill(2, 150, 2, 2, 128, 128, seed=45, h0_std=0.1, kda=True)
    check(gdn, oracle_mod, x, True, True, hT_alias=True, path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("g_steep", [-0.9, -1.5, -2.5, -6.0])
def test_kda_steep_decays(gdn, oracle_mod, g_steep, path):
    """Some key channels decay steeply. The tensor-core prep computes A and P as one product of
    rows decayed to a per-channel anchor while every channel's log-decay spans <= 64 over the
    chunk (-0.9: up to 57.6, exponentials up to e^28.8); steeper chunks anchor at each 16-token
    block's first token while the block spans <= 40 (-1.5: 22.5, -2.5: 37.5) and take the
    diagonal blocks' decays pairwise beyond (-6.0: 90). So this covers every form, each near
    its limit."""
    x = workloads.prefill(2, 150, 2, 2, 128, 128, seed=47, h0_std=0.1, kda=True)
    g = x.g.clone()
    g[..., 5::9] = g_steep                # every ninth channel, from channel 5
    g[:, 70:90, :, 100:] = g_steep        # and a token range of the upper channels
    x.g = g.contiguous()
    check(gdn, oracle_mod, x, False, False, path=path)
    check(gdn, oracle_mod, x, True, True, path=path)


def test_kda_paths_agree_closely(gdn):
    """The tensor-core KDA path splits every fp32 operand into bf16 hi + lo (products keep
    about 16 mantissa bits) and the CUDA-core path multiplies in fp32: on a QDQ-off case their
    outputs agree far inside the oracle bound."""
    x = workloads.prefill(2, 333, 2, 4, 128, 128, seed=46, h0_std=0.1, kda=True)
    o1, h1 = run_gpu(gdn, x, False, False, path="split")
    o2, h2 = run_gpu(gdn, x, False, False, path="fused")
    from helpers import rel
    assert rel(o1.cpu().double().numpy(), o2.cpu().double().numpy()) <= 1e-4
    assert rel(h1.cpu().double().numpy(), h2.cpu().double().numpy()) <= 1e-4


# ---- full-size workloads, sampled (sequence, head) units ---------------------------------

@pytest.mark.parametrize("path", PATHS)
def test_gdn_b4_h16_t4096_d128_sampled(gdn, oracle_mod, path):
    x = workloads.workload("gdn_b4_h16_t4096_d128")
    units = sample_units(4, 16, 16, seed=1)
    check(gdn, oracle_mod, x, True, True, units, path=path)        # the benchmarked configuration
    check(gdn, oracle_mod, x, False, False, units, path=path)      # quantizers off: the 1e-3 bound


@pytest.mark.parametrize("path", PATHS)
def test_gdn_varlen8_hqk16_hv32_d128_sampled(gdn, oracle_mod, path):
    x = workloads.workload("gdn_varlen8_hqk16_hv32_d128")
    lens = np.diff(x.cu_seqlens.numpy())
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    units = sorted(set(sample_units(8, 32, 16, seed=2) + [(longest, 31), (shortest, 0)]))
    check(gdn, oracle_mod, x, True, False, units, path=path)


@pytest.mark.parametrize("path", PATHS)
def test_kda_b2_h32_t8192_d128_sampled(gdn, oracle_mod, path):
    x = workloads.workload("kda_b2_h32_t8192_d128")
    units = sample_units(2, 32, 16, seed=4)
    check(gdn, oracle_mod, x, True, True, units, path=path)


def test_gdn_b4_h16_t4096_d128_quantizers_take_effect(gdn, oracle_mod):
    """The benchmarked configuration is much closer to the oracle with the state and W
    quantizers on than to the same oracle with them off: the QDQ steps really run (the
    per-unit errors with QDQ sit near 1e-4 to 1e-3, the quantization itself moves the result by
    percents)."""
    from helpers import rel
    x = workloads.workload("gdn_b4_h16_t4096_d128")
    units = sample_units(4, 16, 4, seed=8)
    o, hT = run_gpu(gdn, x, True, True)
    o, hT = o.cpu().double().numpy(), hT.cpu().double().numpy()
    on = run_oracle(oracle_mod, x, True, True, units)
    off = oracle_mod.gdn_chunked(x.q, x.k, x.v, x.g, x.beta, x.h0, None, state_qdq=False, w_qdq=False,
                                 unit_mask=mask_for(units, 4, 16))
    ns, hs = (list(t) for t in zip(*units))
    for got, want_on, want_off in ((o[ns, :, hs], on[0][ns, :, hs], off[0][ns, :, hs]),
                                   (hT[ns, hs], on[1][ns, hs], off[1][ns, hs])):
        e_on, e_off = rel(got, want_on), rel(got, want_off)
        assert e_on <= TOL_QDQ and e_off >= 10 * e_on, (e_on, e_off)
