"""fp64 gradient oracle of the gated-delta-rule forward with straight-through state QDQ.

TEST INFRASTRUCTURE ONLY (as the rest of ``oracle/``): the slow, plain reference the CUDA
backward is checked against. Only tests/ and bench.py's CPU leg may import it.

What it differentiates ("Torch GDN/KDA decode QAT with INT8 recurrent state", "Megatron-Core
QAT/QAD workflow" step 4: the recurrent surrogate gradients come from Torch, and the QDQ passes
gradients through unchanged (a straight-through estimator); "GDN state/W QAT foundation": identity straight-through gradients for
QAT): the token recurrence of the forward oracle,
    S_t = a_t S_{t-1} + b_t k_t (v_t - a_t S_{t-1}^T k_t)^T,   o_t = scale S_t^T q_t,
with a_t = exp(g_t) (KDA: row c of S scaled by exp(g_t[c])), and the state QDQ after every 64th
token of a sequence (E4M3 tiles or INT8 blocks). The QDQ forward is the oracle's own fp64 codec;
its backward is the identity. The derivatives themselves come from PyTorch autograd on CPU in
fp64 (a library routine serving as a step), so every gradient is the exact derivative of the
written-out recurrence, with QDQ replaced by the identity in the backward only.
gdn_chunked_grads differentiates the chunked / WY form the same way; it is the only form in which
the W quantizer exists, so it also defines the straight-through gradient with W QDQ on.
"""
from __future__ import annotations

import numpy as np
import torch

from . import int8_block_qdq_f64, tile_qdq_f64


class _StateQdqSte(torch.autograd.Function):
    """Forward: the state codec on S [dk, dv] (E4M3 tiles of 64 columns over all rows, or INT8
    blocks of 32 columns per row), or with codec "w" the W quantizer (one E4M3 tile over a chunk's
    L x dk block). Backward: identity (straight-through)."""

    @staticmethod
    def forward(ctx, S, codec):
        x = S.detach().cpu().numpy()
        if codec == "int8":
            y = int8_block_qdq_f64(x, 32)[0]
        elif codec == "w":   # the W quantizer: one E4M3 tile over the chunk's L x dk block
            y = tile_qdq_f64(x, x.shape[1])[0][0]
        else:
            y = tile_qdq_f64(x, 64)[0][0]
        return torch.from_numpy(np.ascontiguousarray(y)).to(S.dtype)

    @staticmethod
    def backward(ctx, grad):
        return grad, None


def _t(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).clone()
    return torch.as_tensor(np.asarray(x), dtype=torch.float64)


def gdn_recurrent_grads(q, k, v, g, beta, h0=None, cu_seqlens=None, do=None, dhT=None, *, kda=False,
                        state_qdq=False, scale=1.0, codec="e4m3", qdq_period=64, units=None):
    """Gradients of sum(o * do) + sum(hT * dhT) with respect to q, k, v, g, beta and h0, for the
    recurrence above (layouts of the forward oracle: q, k [B, T, Hqk, dk]; v [B, T, Hv, dv];
    g [B, T, Hv] (KDA [B, T, Hv, dk]); beta [B, T, Hv]; h0, hT [N, Hv, dk, dv]; do like o
    [B, T, Hv, dv]). units: a list of (sequence, v-head) pairs to include (the loss then covers only
    their outputs and final states), or None for all. Returns fp64 numpy arrays
    (dq, dk, dv, dg, dbeta, dh0, o, hT)."""
    q, k, v, g, beta = (_t(x).requires_grad_(True) for x in (q, k, v, g, beta))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G = Hv // Hqk
    if cu_seqlens is not None:
        cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        N = len(cu) - 1
        spans = [(0, cu[n], cu[n + 1] - cu[n]) for n in range(N)]
    else:
        N = B
        spans = [(n, 0, T) for n in range(B)]
    h0 = torch.zeros((N, Hv, dk, dv), dtype=torch.float64) if h0 is None else _t(h0)
    h0.requires_grad_(True)
    do = torch.zeros((B, T, Hv, dv), dtype=torch.float64) if do is None else _t(do)
    dhT = None if dhT is None else _t(dhT)
    head_of = torch.arange(Hv) // G   # v-head h reads q / k head h / G
    o_rows, hTs, loss = {}, [], torch.zeros((), dtype=torch.float64)
    keep = None if units is None else set((int(n), int(h)) for n, h in units)
    for n, (b, t0, L) in enumerate(spans):
        for h in range(Hv):
            if keep is not None and (n, h) not in keep:
                hTs.append(torch.zeros((dk, dv), dtype=torch.float64))
                continue
            hq = int(head_of[h])
            S = h0[n, h]
            for t in range(L):
                tok = t0 + t
                kt, qt, vt, bt = k[b, tok, hq], q[b, tok, hq], v[b, tok, h], beta[b, tok, h]
                a = torch.exp(g[b, tok, h])
                Sd = (a[:, None] if kda else a) * S                    # 1. decay
                d = bt * (vt - Sd.t() @ kt)                            # 2-3. delta
                S = Sd + torch.outer(kt, d)                            # 4. update
                o = scale * (S.t() @ qt)                               # 5. output (pre-QDQ state)
                loss = loss + (o * do[b, tok, h]).sum()
                o_rows[(b, tok, h)] = o.detach()
                if state_qdq and (t + 1) % qdq_period == 0:            # 6. state QDQ, identity backward
                    S = _StateQdqSte.apply(S, codec)
            if dhT is not None:
                loss = loss + (S * dhT[n, h]).sum()
            hTs.append(S.detach())
    grads = torch.autograd.grad(loss, [q, k, v, g, beta, h0], allow_unused=True)
    out = [np.zeros(tuple(x.shape)) if gr is None else gr.numpy() for gr, x in zip(grads, (q, k, v, g, beta, h0))]
    o_full = np.zeros((B, T, Hv, dv))
    for (b, tok, h), val in o_rows.items():
        o_full[b, tok, h] = val.numpy()
    hT = torch.stack(hTs).reshape(N, Hv, dk, dv).numpy()
    return (*out, o_full, hT)


def gdn_chunked_grads(q, k, v, g, beta, h0=None, cu_seqlens=None, do=None, dhT=None, *, kda=False,
                      state_qdq=False, w_qdq=False, scale=1.0, codec="e4m3", chunk=64):
    """The same gradients through the chunked / WY form of the forward ("GDN state/W QAT
    foundation", "What does this PR do?": W is the WY-transformed key block, quantized once per
    chunk, and both quantizers pass gradients straight through). Per chunk of L tokens entering
    with state S0, gam the prefix sums of g inside the chunk (KDA: per key channel):
        A[r][i] = beta_r sum_c k_r[c] k_i[c] exp(gam_r[c] - gam_i[c])  (i < r),  T = (I + A)^-1,
        W = T (beta exp(gam) K) [W <- QDQ(W), one L x dk E4M3 tile, when w_qdq],  U = T (beta V),
        Delta = U - W S0,  o = scale (exp(gam) Q S0 + P Delta),
        P[r][i] = sum_c q_r[c] k_i[c] exp(gam_r[c] - gam_i[c])  (i <= r),
        S1 = exp(gam_L) S0 + (K exp(gam_L - gam))^T Delta,  S1 <- QDQ(S1) on a 64-token boundary.
    Without W QDQ this is the token recurrence rewritten, so its gradients equal
    gdn_recurrent_grads'; with W QDQ it is the only form in which that quantizer exists.
    PyTorch autograd in fp64 on CPU supplies the derivatives. Same layouts and return values as
    gdn_recurrent_grads (all units)."""
    q, k, v, g, beta = (_t(x).requires_grad_(True) for x in (q, k, v, g, beta))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G = Hv // Hqk
    if cu_seqlens is not None:
        cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        N = len(cu) - 1
        spans = [(0, cu[n], cu[n + 1] - cu[n]) for n in range(N)]
    else:
        N = B
        spans = [(n, 0, T) for n in range(B)]
    h0 = torch.zeros((N, Hv, dk, dv), dtype=torch.float64) if h0 is None else _t(h0)
    h0.requires_grad_(True)
    do = torch.zeros((B, T, Hv, dv), dtype=torch.float64) if do is None else _t(do)
    dhT = None if dhT is None else _t(dhT)
    loss = torch.zeros((), dtype=torch.float64)
    o_rows, hTs = {}, []
    for n, (b, t0, L_seq) in enumerate(spans):
        for h in range(Hv):
            hq = h // G
            S = h0[n, h]
            for c0 in range(0, L_seq, chunk):
                L = min(chunk, L_seq - c0)
                rows = slice(t0 + c0, t0 + c0 + L)
                Kc, Qc, Vc, bc = k[b, rows, hq], q[b, rows, hq], v[b, rows, h], beta[b, rows, h]
                gc = g[b, rows, h]
                gam = torch.cumsum(gc, dim=0)
                gam2 = gam if kda else gam[:, None].expand(L, dk)               # [L, dk]
                incl = torch.tril(torch.ones((L, L), dtype=torch.bool))
                diff = gam2[:, None, :] - gam2[None, :, :]                    # [r, i, c]
                E = torch.exp(torch.where(incl[:, :, None], diff, torch.zeros_like(diff)))
                E = E * incl[:, :, None]                                     # exp(gam_r - gam_i), i <= r
                strict = torch.tril(torch.ones((L, L), dtype=torch.float64), diagonal=-1)
                A = bc[:, None] * (Kc[:, None, :] * Kc[None, :, :] * E).sum(-1) * strict
                Tm = torch.linalg.inv(torch.eye(L, dtype=torch.float64) + A)
                W = Tm @ (bc[:, None] * torch.exp(gam2) * Kc)
                U = Tm @ (bc[:, None] * Vc)
                if w_qdq:
                    W = _StateQdqSte.apply(W, "w")
                Dl = U - W @ S
                P = (Qc[:, None, :] * Kc[None, :, :] * E).sum(-1)
                O = scale * ((Qc * torch.exp(gam2)) @ S + P @ Dl)
                loss = loss + (O * do[b, rows, h]).sum()
                for r in range(L):
                    o_rows[(b, t0 + c0 + r, h)] = O[r].detach()
                gl = gam2[L - 1]
                S = torch.exp(gl)[:, None] * S + (Kc * torch.exp(gl[None, :] - gam2)).t() @ Dl
                if state_qdq and (c0 + L) % 64 == 0:
                    S = _StateQdqSte.apply(S, codec)
            if dhT is not None:
                loss = loss + (S * dhT[n, h]).sum()
            hTs.append(S.detach())
    grads = torch.autograd.grad(loss, [q, k, v, g, beta, h0], allow_unused=True)
    out = [np.zeros(tuple(x.shape)) if gr is None else gr.numpy() for gr, x in zip(grads, (q, k, v, g, beta, h0))]
    o_full = np.zeros((B, T, Hv, dv))
    for (b, tok, h), val in o_rows.items():
        o_full[b, tok, h] = val.numpy()
    hT = torch.stack(hTs).reshape(N, Hv, dk, dv).numpy()
    return (*out, o_full, hT)
