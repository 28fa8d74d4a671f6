"""Seeded synthetic inputs for the chunked gated-delta-rule forward and its decode step.

This module is the one piece shared by the CUDA library's tests/benchmark and the oracle:
it only draws random numbers (CPU ``torch.Generator``) and holds none of the method's
arithmetic. Distributions follow the workloads the method is exercised on:

* q, k: N(0, 1) -> bf16 -> L2-normalised over the head dimension in fp32 -> bf16
* v: N(0, 1) -> bf16
* beta = sigmoid(N(0, 1)) fp32; g = log(alpha), alpha = sigmoid(N(3, 1)) fp32
  (per head-token; per head-token-key-channel for KDA)
* h0: N(0, std) fp32 or absent (zeros)

All tensors are CPU tensors in the head-last layout the library uses:
q, k [B, T, Hqk, dk]; v [B, T, Hv, dv]; g [B, T, Hv] (KDA [B, T, Hv, dk]); beta [B, T, Hv];
h0 [N, Hv, dk, dv]; varlen packs N sequences on the T axis of B = 1 with int32 cu_seqlens.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    kda: bool = False
    state_qdq: bool = True
    w_qdq: bool = False
    name: str = ""
    # prefill -> decode handoff: per sequence, the tokens that run as chunked prefill (the rest
    # run as decode steps); None = plain chunked prefill
    prefill_lengths: Optional[list] = None
    backward: bool = False   # the workload times the backward pass

    @property
    def shape(self):
        B, T, Hqk, dk = self.q.shape
        return dict(B=B, T=T, Hqk=Hqk, Hv=self.v.shape[2], dk=dk, dv=self.v.shape[3],
                    N=(self.cu_seqlens.numel() - 1) if self.cu_seqlens is not None else B)

    def tokens(self) -> int:
        return self.q.shape[0] * self.q.shape[1]


@dataclass
class QdqInputs:
    x: torch.Tensor      # [lead, rows, cols] fp32
    tile_cols: int       # E4M3: a tile is all rows x tile_cols columns; INT8: a block is tile_cols columns of a row
    name: str = ""
    codec: str = "e4m3"


@dataclass
class DecodeInputs:
    q: torch.Tensor      # [steps, N, Hqk, dk] bf16
    k: torch.Tensor      # [steps, N, Hqk, dk] bf16
    v: torch.Tensor      # [steps, N, Hv, dv] bf16
    g: torch.Tensor      # [steps, N, Hv] fp32 (KDA [steps, N, Hv, dk])
    beta: torch.Tensor   # [steps, N, Hv] fp32
    state: torch.Tensor  # [N, Hv, dk, dv] fp32
    kda: bool = False
    state_qdq: bool = True
    name: str = ""
    codec: str = "e4m3"  # state QDQ format: "e4m3" tiles or "int8" blocks


def _normal(gen, shape, mean=0.0, std=1.0):
    x = torch.empty(shape, dtype=torch.float32)
    x.normal_(mean=mean, std=std, generator=gen)
    return x


def _unit_bf16(gen, shape):
    x = _normal(gen, shape).to(torch.bfloat16).to(torch.float32)
    x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return x.to(torch.bfloat16)


def prefill(B, T, Hqk, Hv, dk, dv, *, seed, kda=False, h0_std=None, seqlens=None,
            state_qdq=True, w_qdq=False, name="") -> PrefillInputs:
    """Dense (seqlens None) or packed varlen (B must be 1) prefill inputs."""
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if seqlens is not None:
        assert B == 1
        lens = torch.as_tensor(seqlens, dtype=torch.int64)
        cu = torch.zeros(lens.numel() + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
        T = int(cu[-1])
    N = (cu.numel() - 1) if cu is not None else B
    q = _unit_bf16(gen, (B, T, Hqk, dk))
    k = _unit_bf16(gen, (B, T, Hqk, dk))
    v = _normal(gen, (B, T, Hv, dv)).to(torch.bfloat16)
    beta = torch.sigmoid(_normal(gen, (B, T, Hv)))
    gshape = (B, T, Hv, dk) if kda else (B, T, Hv)
    g = torch.log(torch.sigmoid(_normal(gen, gshape, mean=3.0)))
    h0 = _normal(gen, (N, Hv, dk, dv), std=h0_std) if h0_std else None
    return PrefillInputs(q, k, v, g.contiguous(), beta.contiguous(), h0, cu, kda=kda,
                         state_qdq=state_qdq, w_qdq=w_qdq, name=name)


def _backward(x: PrefillInputs) -> PrefillInputs:
    x.backward = True
    return x


def handoff(B, T, P, Hqk, Hv, dk, dv, *, seed, kda=False, name="") -> PrefillInputs:
    """Dense batch whose sequences run their first P tokens as chunked prefill and the rest as
    decode steps; state and W QDQ on, h0 = 0."""
    x = prefill(B, T, Hqk, Hv, dk, dv, seed=seed, kda=kda, h0_std=None, state_qdq=True, w_qdq=True, name=name)
    x.prefill_lengths = [P] * B
    return x


def varlen_lengths(n_seqs, max_len, seed):
    """Sequence lengths ~ U[1, max_len] drawn from the workload's own seed."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(1, max_len + 1, (n_seqs,), generator=gen).tolist()


def decode(steps, N, H, dk, dv, *, seed, kda=False, state_std=0.05, state_qdq=True, name="",
           codec="e4m3") -> DecodeInputs:
    gen = torch.Generator().manual_seed(seed)
    state = _normal(gen, (N, H, dk, dv), std=state_std)
    q = _unit_bf16(gen, (steps, N, H, dk))
    k = _unit_bf16(gen, (steps, N, H, dk))
    v = _normal(gen, (steps, N, H, dv)).to(torch.bfloat16)
    beta = torch.sigmoid(_normal(gen, (steps, N, H)))
    gshape = (steps, N, H, dk) if kda else (steps, N, H)
    g = torch.log(torch.sigmoid(_normal(gen, gshape, mean=3.0)))
    return DecodeInputs(q, k, v, g.contiguous(), beta.contiguous(), state, kda=kda,
                        state_qdq=state_qdq, name=name, codec=codec)


def qdq(lead, rows, cols, tile_cols, *, seed, std=0.05, name="", codec="e4m3") -> QdqInputs:
    """Standalone QDQ input: a state-shaped fp32 tensor."""
    gen = torch.Generator().manual_seed(seed)
    return QdqInputs(_normal(gen, (lead, rows, cols), std=std), tile_cols, name=name, codec=codec)


# --- the named workloads --------------------------------------------------------------

WORKLOADS = {
    # small parity case: 4 chunks of 64, state QDQ on, W QDQ off, h0 = 0
    "gdn_b1_h2_t256_d64": lambda: prefill(1, 256, 2, 2, 64, 64, seed=0, state_qdq=True, w_qdq=False,
                                          name="gdn_b1_h2_t256_d64"),
    # the throughput workload: state + W QDQ, h0 ~ N(0, 0.1)
    "gdn_b4_h16_t4096_d128": lambda: prefill(4, 4096, 16, 16, 128, 128, seed=1, h0_std=0.1, state_qdq=True,
                                             w_qdq=True, name="gdn_b4_h16_t4096_d128"),
    # varlen: 8 sequences of U[1, 8192] tokens, GQA 16 q/k heads -> 32 v heads
    "gdn_varlen8_hqk16_hv32_d128": lambda: prefill(1, 0, 16, 32, 128, 128, seed=2, h0_std=0.1,
                                                   seqlens=varlen_lengths(8, 8192, seed=2), state_qdq=True,
                                                   w_qdq=False, name="gdn_varlen8_hqk16_hv32_d128"),
    # decode: 512 sequences x 32 heads, 64 single-token steps, QDQ on every write
    "gdn_decode_n512_h32_d128_s64": lambda: decode(64, 512, 32, 128, 128, seed=3, state_std=0.05,
                                                   name="gdn_decode_n512_h32_d128_s64"),
    # the backward of the prefill benchmark's shape (state QDQ straight through; no W QDQ, whose
    # straight-through gradient needs the chunked form)
    "gdn_bwd_b4_h16_t4096_d128": lambda: _backward(prefill(4, 4096, 16, 16, 128, 128, seed=1, h0_std=0.1,
                                                           state_qdq=True, w_qdq=False,
                                                           name="gdn_bwd_b4_h16_t4096_d128")),
    # the backward of the KDA benchmark's shape (state QDQ straight through, no W QDQ)
    "kda_bwd_b2_h32_t8192_d128": lambda: _backward(prefill(2, 8192, 32, 32, 128, 128, seed=4, kda=True, h0_std=0.1,
                                                           state_qdq=True, w_qdq=False,
                                                           name="kda_bwd_b2_h32_t8192_d128")),
    # the decode workload with the INT8 block-32 state codec
    "gdn_decode_int8_n512_h32_d128_s64": lambda: decode(64, 512, 32, 128, 128, seed=3, state_std=0.05,
                                                        name="gdn_decode_int8_n512_h32_d128_s64", codec="int8"),
    # standalone INT8 block QDQ over the same decode-sized state tensor, 32-column blocks per key row
    "int8_state_n512_h32_d128": lambda: qdq(512 * 32, 128, 128, 32, seed=5, name="int8_state_n512_h32_d128",
                                            codec="int8"),
    # standalone tile QDQ over a decode-sized state tensor: 16384 x [128 x 128], 64-column tiles
    "qdq_state_n512_h32_d128": lambda: qdq(512 * 32, 128, 128, 64, seed=5, name="qdq_state_n512_h32_d128"),
    # prefill -> decode handoff, the QAT/QAD workflow's example shape (128-token sequences, the
    # first 64 tokens as chunked prefill, the last 64 as decode steps) over 256 sequences x 16
    # heads; state + W QDQ, h0 = 0 (a training sequence starts from an empty state)
    "handoff_n256_t128_p64_h16_d128": lambda: handoff(256, 128, 64, 16, 16, 128, 128, seed=6,
                                                      name="handoff_n256_t128_p64_h16_d128"),
    # KDA: per-key-channel decay, state + W QDQ, h0 = 0
    "kda_b2_h32_t8192_d128": lambda: prefill(2, 8192, 32, 32, 128, 128, seed=4, kda=True, state_qdq=True,
                                             w_qdq=True, name="kda_b2_h32_t8192_d128"),
}


def workload(name: str):
    return WORKLOADS[name]()
