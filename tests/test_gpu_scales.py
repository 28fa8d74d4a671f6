"""The optional final-state QDQ scales of the chunk and handoff calls (gdn_chunk_args.state_scales).

Where a sequence's final state was QDQ'd (its last token was a 64th token; for the handoff, it had
decode tokens), hT must be exactly code x scale: hT / scale lies on the codec's grid and the tile's
(block's) largest element maps to the codec's largest code (448 E4M3, 127 INT8). Elsewhere the
scale is 0. Checked on every chunk path (tensor-core split, fused / CUDA-core, dk = 64), for GDN
and KDA, both codecs, and the handoff.
"""
import numpy as np
import pytest
import torch

from fp8_state_qat_gb300 import workloads
from helpers import to_cuda

pytestmark = pytest.mark.gpu

LENS = [0, 1, 64, 100, 128, 192]


def e4m3_grid(y):
    """|y| <= 448 and y an E4M3 value (3 mantissa bits; subnormal spacing 2^-9)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -9)))
    q = 2.0 ** (np.maximum(e, -6) - 3)
    return (a <= 448 * (1 + 1e-6)) & (np.abs(a / q - np.round(a / q)) <= 1e-5 * np.maximum(a / q, 1))


def check_scales(hT, sc, lens, codec, dk, dv, P=None):
    hT = hT.cpu().double().numpy()
    sc = sc.cpu().double().numpy()
    N, Hv = hT.shape[:2]
    for n in range(N):
        qd = (lens[n] > P[n]) if P is not None else (lens[n] > 0 and lens[n] % 64 == 0)
        for h in range(Hv):
            if codec == "e4m3":
                for t in range(dv // 64):
                    s = sc[n, h, t]
                    if not qd:
                        assert s == 0.0
                        continue
                    y = hT[n, h, :, 64 * t:64 * t + 64] / s
                    assert s > 0 and e4m3_grid(y).all() and abs(np.abs(y).max() - 448.0) <= 448e-6, (n, h, t)
            else:
                for r in range(dk):
                    for b in range(dv // 32):
                        s = sc[n, h, r, b]
                        if not qd:
                            assert s == 0.0
                            continue
                        y = hT[n, h, r, 32 * b:32 * b + 32] / s
                        c = np.round(y)
                        assert s > 0 and np.all(np.abs(y - c) <= 1e-5 * np.maximum(np.abs(c), 1)), (n, h, r, b)
                        assert np.abs(c).max() == 127.0


def scales_tensor(N, Hv, dk, dv, codec):
    shape = (N, Hv, dv // 64) if codec == "e4m3" else (N, Hv, dk, dv // 32)
    return torch.full(shape, -1.0, device="cuda")   # every entry must be written


@pytest.mark.parametrize("codec", ["e4m3", "int8"])
@pytest.mark.parametrize("kda", [False, True])
@pytest.mark.parametrize("path,dk,dv", [("split", 128, 128), ("fused", 128, 128), ("split", 128, 64), ("split", 64, 128)])
def test_chunk_state_scales(gdn, codec, kda, path, dk, dv):
    x = workloads.prefill(1, 0, 2, 2, dk, dv, seed=70 + dk + dv + kda, kda=kda, h0_std=0.1, seqlens=LENS)
    c = to_cuda(x)
    fn = gdn.kda_chunk_fwd if kda else gdn.gdn_chunk_fwd
    ws = torch.empty(256, dtype=torch.uint8, device="cuda") if path == "fused" else None
    sc = scales_tensor(len(LENS), 2, dk, dv, codec)
    o, hT = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, state_qdq=True, w_qdq=True,
               workspace=ws, codec=codec, state_scales=sc)
    torch.cuda.synchronize()
    check_scales(hT, sc, LENS, codec, dk, dv)


@pytest.mark.parametrize("codec", ["e4m3", "int8"])
@pytest.mark.parametrize("kda", [False, True])
def test_handoff_state_scales(gdn, codec, kda):
    P = [0, 1, 64, 37, 128, 150]
    x = workloads.prefill(1, 0, 2, 2, 128, 128, seed=77 + kda, kda=kda, h0_std=0.1, seqlens=LENS)
    c = to_cuda(x)
    fn = gdn.kda_prefill_decode_fwd if kda else gdn.gdn_prefill_decode_fwd
    P = [min(p, L) for p, L in zip(P, LENS)]
    sc = scales_tensor(len(LENS), 2, 128, 128, codec)
    o, hT = fn(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], x.cu_seqlens, P, state_qdq=True, w_qdq=True,
               codec=codec, state_scales=sc)
    torch.cuda.synchronize()
    check_scales(hT, sc, LENS, codec, 128, 128, P=P)


def test_state_scales_need_the_state_quantizer(gdn):
    x = workloads.prefill(1, 64, 1, 1, 128, 128, seed=79)
    c = to_cuda(x)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_chunk_fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], None, None, state_qdq=False,
                          state_scales=torch.zeros((1, 1, 2), device="cuda"))
