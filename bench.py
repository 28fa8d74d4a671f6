#!/usr/bin/env python
"""Throughput of the chunked gated-delta-rule forward with FP8 E4M3 state and W QDQ.

Workload: B=4, H=16 (q/k and v heads), T=4096, dk=dv=128, state QDQ + W QDQ, h0 ~ N(0, 0.1),
synthetic seeded inputs (fp8_state_qat_gb300.workloads). One step = one gdn_chunk_fwd call
over the whole batch; inputs resident in HBM (two alternating input sets of 346 MB each,
larger than the 129 MB L2). Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

N > 1 (launched by torch.distributed.run): every rank runs its own replica of the workload on
its own GPU (the path has no exchange step; weak scaling), timing is max over ranks.
--impl reference times the fp64 CPU oracle instead (rank 0 only), on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "gdn_b4_h16_t4096_d128"
METRIC = "GDN chunked-prefill tokens/s (B4 H16 T4096 d128, FP8 state QDQ); % of roofline"
UNIT = "tokens/s"


def algorithmic(x):
    """Counted bytes and FLOPs of one forward over the workload. Bytes: q, k (per q/k head),
    v in bf16, g and beta in fp32, o in fp32, h0 read and hT write in fp32. FLOPs per
    token-head: 2 [C dk (K K^T) + C dk (Q K^T) + C (dk + dv) (T [beta Gam K | beta V])
    + 3 dk dv (W S, Q S, K^T Delta) + C dv (P Delta)] + C^2 / 3 (solve), C = 64."""
    s = x.shape
    tok = x.tokens()
    C = 64
    by = tok * (s["Hqk"] * 2 * s["dk"] * 2 + s["Hv"] * (2 * s["dv"] + 8 + 4 * s["dv"]))
    by += (2 if x.h0 is not None else 1) * s["N"] * s["Hv"] * s["dk"] * s["dv"] * 4
    fl_th = 2 * (C * s["dk"] * 2 + C * (s["dk"] + s["dv"]) + 3 * s["dk"] * s["dv"] + C * s["dv"]) + C * C / 3
    if x.prefill_lengths is None:
        return by, fl_th * tok * s["Hv"]
    # prefill -> decode handoff: the decode tokens cost 7 dk dv each (decay, S^T k, k d^T, S^T q)
    pre = sum(x.prefill_lengths)
    return by, (fl_th * pre + 7 * s["dk"] * s["dv"] * (tok - pre)) * s["Hv"]


def alu_peak(dev, torch, sm_max_mhz):
    """fp32 CUDA-core peak in TFLOP/s from unit counts and clocks: SMs x 128 fp32 lanes x 2 flop
    (an FMA) x the maximum SM clock (the sampled clocks.max.sm, else 2070 MHz)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = sm_max_mhz or 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sms} SMs x 128 fp32 lanes x 2 flop x {mhz:.0f} MHz"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# the sources that build the benchmark step's two kernels (and the host code that launches them)
PREFILL_SOURCES = ("chunk_prep.cu", "chunk_chain.cu", "tma_maps.cu", "gdnqat_api.cu", "common.cuh", "tc_common.cuh",
                   "tc_epilogue.cuh", "kernels.h")
# per workload: its ncu summary and the sources of the kernels a step launches
PROFILES = {
    "gdn_b4_h16_t4096_d128": ("chunk_fwd_gdn_b4_h16_t4096_d128.md", PREFILL_SOURCES),
    "gdn_decode_n512_h32_d128_s64": ("decode_gdn_decode_n512_h32_d128_s64.md",
                                     ("decode.cu", "gdnqat_api.cu", "common.cuh", "kernels.h")),
    "qdq_state_n512_h32_d128": ("tile_qdq_qdq_state_n512_h32_d128.md",
                                ("qdq.cu", "gdnqat_api.cu", "common.cuh", "tc_epilogue.cuh", "tc_common.cuh", "kernels.h")),
    "gdn_varlen8_hqk16_hv32_d128": ("chunk_fwd_gdn_varlen8_hqk16_hv32_d128.md", PREFILL_SOURCES),
    "handoff_n256_t128_p64_h16_d128": ("handoff_n256_t128_p64_h16_d128.md", PREFILL_SOURCES + ("handoff.cu",)),
    "gdn_decode_int8_n512_h32_d128_s64": ("decode_gdn_decode_int8_n512_h32_d128_s64.md",
                                          ("decode.cu", "gdnqat_api.cu", "common.cuh", "kernels.h")),
    "int8_state_n512_h32_d128": ("int8_block_qdq_int8_state_n512_h32_d128.md",
                                 ("qdq.cu", "gdnqat_api.cu", "common.cuh", "tc_epilogue.cuh", "tc_common.cuh",
                                  "kernels.h")),
    "gdn_bwd_b4_h16_t4096_d128": ("chunk_bwd_gdn_bwd_b4_h16_t4096_d128.md",
                                  ("backward.cu", "gdnqat_api.cu", "common.cuh", "kernels.h")),
    "kda_bwd_b2_h32_t8192_d128": ("chunk_bwd_kda_bwd_b2_h32_t8192_d128.md",
                                  ("backward.cu", "gdnqat_api.cu", "common.cuh", "kernels.h")),
    "kda_b2_h32_t8192_d128": ("chunk_fwd_kda_b2_h32_t8192_d128.md",
                              ("chunk_prep_kda.cu", "chunk_chain_kda.cu", "tma_maps.cu", "gdnqat_api.cu", "common.cuh",
                               "tc_common.cuh", "tc_epilogue.cuh", "kernels.h")),
}


def code_only(text):
    """C / CUDA source without its comments and trailing blanks: what the compiler sees (the
    sources have no string literal holding a comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(sources=PREFILL_SOURCES):
    """Hash of the code (comments excluded) of the sources that build a step's kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_state_qat_gb300", "csrc")
    for name in sorted(sources):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload=WORKLOAD):
    """DRAM bytes per launch from the workload's committed ncu summary, if it was taken on the
    current sources of its kernels (else None)."""
    if workload not in PROFILES:
        return None
    name, sources = PROFILES[workload]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash(sources):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return None
        inside = [r for t, r in self.rows if self.t0 and self.t1 and self.t0 - 0.15 <= t <= self.t1 + 0.15]
        rows = inside or [r for _, r in self.rows]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "in_timed_region": bool(inside)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The slowest replica's figure: every rank's x reduced with MAX (a collective when world > 1;
    it runs on the ranks' NCCL group on GPUs, on gloo in the CPU tests)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput of `world` replicas (weak scaling): every rank's units over the
    slowest rank's milliseconds."""
    return world * units_per_rank / (ms * 1e-3)


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (model name, else implementer / part), and the ISA."""
    import platform
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "CPU part"):
            for line in info.splitlines():
                if line.startswith(key):
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                name = f"{key} {name}" if key == "CPU part" else name
                break
    except OSError:
        pass
    return f"{platform.machine()} {name}".strip()


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_inputs(x, t_tokens):
    """The workload's first t_tokens tokens as contiguous fp32/fp64 numpy arrays (converted
    once, outside any timed region)."""
    import numpy as np

    sl = slice(0, t_tokens)
    f = lambda t: np.ascontiguousarray(t[:, sl].float().numpy())
    return (f(x.q), f(x.k), f(x.v), f(x.g), f(x.beta),
            None if x.h0 is None else np.ascontiguousarray(x.h0.double().numpy()))


def oracle_sample(x, arrays, units, threads):
    """Chunked fp64 oracle (state + W QDQ) on the first `units` (sequence, head) units of the
    prepared arrays. Returns (seconds, tokens in the metric's unit)."""
    import numpy as np

    import oracle

    s = x.shape
    mask = np.zeros((s["N"], s["Hv"]), np.uint8)
    mask.reshape(-1)[:units] = 1
    q, k, v, g, beta, h0 = arrays
    t = time.perf_counter()
    oracle.gdn_chunked(q, k, v, g, beta, h0, None, state_qdq=x.state_qdq, w_qdq=x.w_qdq, unit_mask=mask,
                       threads=threads)
    dt = time.perf_counter() - t
    # a (sequence, head) unit over L tokens is 1/Hv of the work of L batch tokens
    return dt, units * q.shape[1] / s["Hv"]


def cpu_baseline(x, target_s=15.0):
    """Time the oracle as it stands on all host cores on a bounded sample (~10-30 s of CPU work)."""
    import oracle

    oracle.build()
    cores = cpu_cores()
    s = x.shape
    total_units = s["N"] * s["Hv"]
    dt1, _ = oracle_sample(x, oracle_inputs(x, 512), 1, 1)      # calibrate: one unit, 512 tokens, one thread
    per_unit_full = dt1 * s["T"] / 512
    units = max(1, min(total_units, int(target_s / max(per_unit_full, 1e-6))))
    dt, toks = oracle_sample(x, oracle_inputs(x, s["T"]), units, cores)
    return {"value": toks / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{units} of {total_units} (sequence, head) units x all {s['T']} tokens, chunked fp64 "
                      f"oracle with state+W QDQ, {cores} threads, {dt:.2f} s wall",
            "single_core_value": (512 / s["Hv"]) / dt1, "cpu": cpu_model()}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from fp8_state_qat_gb300 import workloads

    oracle.build()
    x = workloads.workload(WORKLOAD)
    cores = cpu_cores()
    s = x.shape
    budget = 150.0 / max(1, args.steps + args.warmup)        # seconds per step: whole run in a few minutes
    dt1, _ = oracle_sample(x, oracle_inputs(x, 64), 1, 1)
    per_unit_tok = dt1 / 64
    units = max(1, min(s["N"] * s["Hv"], cores))
    t_tok = int(budget * cores / max(units * per_unit_tok, 1e-9)) // 64 * 64
    t_tok = max(64, min(s["T"], t_tok))
    arrays = oracle_inputs(x, t_tok)
    for _ in range(args.warmup):
        oracle_sample(x, arrays, units, cores)
    secs, toks = 0.0, 0.0
    for _ in range(args.steps):
        dt, tk = oracle_sample(x, arrays, units, cores)
        secs += dt
        toks += tk
    value = toks / secs
    sample = (f"per step {units} (sequence, head) units x first {t_tok} tokens of the workload, chunked fp64 "
              f"oracle with state+W QDQ on {cores} host threads")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": 4, "H": 16, "T": 4096, "dk": 128, "dv": 128,
                       "state_qdq": True, "w_qdq": True, "parallelism": "none (host threads)"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def decode_bytes(d):
    """Counted bytes of one decode step: state read + write (fp32), q, k (per q/k head), v
    (bf16), g, beta (fp32; KDA g per key channel), o (fp32)."""
    _, N, Hqk, dk = d.q.shape
    Hv, dv = d.v.shape[2], d.v.shape[3]
    per_head = 2 * 4 * dk * dv + 2 * dv + 4 * (dk if d.kda else 1) + 4 + 4 * dv
    return N * Hv * per_head + N * Hqk * 2 * 2 * dk


class PrefillCase:
    def __init__(self, x, dev, torch, gdn):
        self.x, self.dev, self.torch, self.gdn = x, dev, torch, gdn
        s = self.s = x.shape
        self.tokens = x.tokens()
        self.bytes, self.flops = algorithmic(x)
        if x.kda:
            self.bytes += self.tokens * s["Hv"] * 4 * (s["dk"] - 1)
        self.handoff = x.prefill_lengths is not None
        if self.handoff:
            self.fn = gdn.kda_prefill_decode_fwd if x.kda else gdn.gdn_prefill_decode_fwd
        else:
            self.fn = gdn.kda_chunk_fwd if x.kda else gdn.gdn_chunk_fwd
        self.sets = [self.resident(), self.resident()]
        self.cu = x.cu_seqlens
        # dk = 128 with the full workspace: a parallel prep kernel, then the state chain (and for
        # the handoff the decode-token kernel)
        self.launches = (2 if s["dk"] == 128 else 1) + (1 if self.handoff else 0)

    def scope(self):
        if self.launches == 1:
            return "one step = one kernel launch"
        kernels = ["chunk_prep_kda_kernel", "chunk_chain_kda_kernel"] if self.x.kda else \
            ["chunk_prep_kernel", "chunk_chain_kernel"]
        if self.s["dk"] != 128:
            kernels = ["chunk_simt_kernel"]
        if self.handoff:
            kernels.append("handoff_suffix_kernel")
        return f"one step = {' + '.join(kernels)}; achieved is over all of them"

    def workspace_bytes(self):
        if self.handoff:
            return self.gdn.prefill_decode_workspace_bytes(self.x.q.shape, self.x.v.shape, self.cu,
                                                           state_qdq=self.x.state_qdq, w_qdq=self.x.w_qdq,
                                                           kda=self.x.kda)
        return self.gdn.chunk_workspace_bytes(self.x.q.shape, self.x.v.shape, self.cu, state_qdq=self.x.state_qdq,
                                              w_qdq=self.x.w_qdq, kda=self.x.kda)

    def resident(self):
        x, s, dev, torch = self.x, self.s, self.dev, self.torch
        return dict(q=x.q.to(dev), k=x.k.to(dev), v=x.v.to(dev), g=x.g.to(dev), beta=x.beta.to(dev),
                    h0=None if x.h0 is None else x.h0.to(dev),
                    o=torch.empty((s["B"], s["T"], s["Hv"], s["dv"]), device=dev),
                    hT=torch.empty((s["N"], s["Hv"], s["dk"], s["dv"]), device=dev))

    def step(self, i, ws, stream):
        b = self.sets[i & 1]
        if self.handoff:
            self.fn(b["q"], b["k"], b["v"], b["g"], b["beta"], b["h0"], self.cu, self.x.prefill_lengths,
                    state_qdq=self.x.state_qdq, w_qdq=self.x.w_qdq, o=b["o"], hT=b["hT"], workspace=ws, stream=stream)
            return
        self.fn(b["q"], b["k"], b["v"], b["g"], b["beta"], b["h0"], self.cu, state_qdq=self.x.state_qdq,
                w_qdq=self.x.w_qdq, o=b["o"], hT=b["hT"], workspace=ws, stream=stream)

    def host(self):
        x = self.x
        inp = dict(q=x.q, k=x.k, v=x.v, g=x.g, beta=x.beta)
        if x.h0 is not None:
            inp["h0"] = x.h0
        self.h_in = {k: t.pin_memory() for k, t in inp.items()}
        b = self.sets[0]
        self.h_out = [{k: self.torch.empty(b[k].shape, dtype=self.torch.float32).pin_memory() for k in ("o", "hT")}
                      for _ in range(2)]
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * 4 for t in self.h_out[0].values()))

    def h2d(self, slot):   # on the current stream
        for k, t in self.h_in.items():
            self.sets[slot][k].copy_(t, non_blocking=True)

    def run(self, slot, ws, stream):
        self.step(slot, ws, stream)

    def d2h(self, slot):
        for k, t in self.h_out[slot].items():
            t.copy_(self.sets[slot][k], non_blocking=True)

    def config(self):
        s, x = self.s, self.x
        c = {"workload": x.name, "B": s["B"], "T": s["T"], "Hqk": s["Hqk"], "Hv": s["Hv"], "dk": s["dk"],
             "dv": s["dv"], "state_qdq": x.state_qdq, "w_qdq": x.w_qdq, "kda": x.kda,
             "h0": "N(0,0.1)" if x.h0 is not None else "zeros"}
        if self.cu is not None:
            c["seqlens"] = self.cu.diff().tolist()
        if self.handoff:
            pl = sorted(set(x.prefill_lengths))
            c["prefill_lengths"] = pl[0] if len(pl) == 1 else x.prefill_lengths
        return c


class BwdCase(PrefillCase):
    """One step = one gdn_chunk_bwd over the workload (the gradients of <o, dout> for the forward
    with straight-through state QDQ); inputs and dout resident, two alternating sets."""

    def __init__(self, x, dev, torch, gdn):
        super().__init__(x, dev, torch, gdn)
        s = self.s
        gen = torch.Generator().manual_seed(11)
        self.dout_h = torch.randn((s["B"], s["T"], s["Hv"], s["dv"]), generator=gen)
        for b in self.sets:
            b["dout"] = self.dout_h.to(dev)
        self.fn = gdn.kda_chunk_bwd if x.kda else gdn.gdn_chunk_bwd
        tok, Hv, Hqk, dk, dv = self.tokens, s["Hv"], s["Hqk"], s["dk"], s["dv"]
        gk = dk if x.kda else 1
        # in: q, k (per q/k head), v, g, beta, dout, h0; out: dq, dk (per q/k head), dv, dg, dbeta, dh0
        self.bytes = tok * (Hqk * 2 * dk * 2 + Hv * (2 * dv + 4 * gk + 4 + 4 * dv)) + \
            tok * (Hqk * 2 * dk * 4 + Hv * (4 * dv + 4 * gk + 4)) + \
            (2 if x.h0 is not None else 1) * s["N"] * Hv * dk * dv * 4
        # per token and state element: the forward step that rebuilds the state (decay 1, S^T k 2,
        # k d^T 2) and the backward step (P' 1, u 2, dS += q do^T 2, du 2, S 2, the four row sums
        # 8, dP' 2, dS_{t-1} 1); the kernel's extra recomputes are not counted
        self.flops = tok * Hv * (5 + 20) * dk * dv
        self.launches = 5   # the backward kernel and the sums of the dq, dk, dbeta, dg partials
        self.bound = "alu"  # fp32 arithmetic on the CUDA cores (issue-bound, not DRAM-bound)

    def scope(self):
        return "one step = chunk_bwd_kernel + 4 partial-sum launches (sum_parts4_kernel); achieved is over all of them"

    def workspace_bytes(self):
        return self.gdn.chunk_bwd_workspace_bytes(self.x.q.shape, self.x.v.shape, self.cu, kda=self.x.kda)

    def step(self, i, ws, stream):
        b = self.sets[i & 1]
        b["grads"] = self.fn(b["q"], b["k"], b["v"], b["g"], b["beta"], b["h0"], self.cu, b["dout"],
                             state_qdq=self.x.state_qdq, workspace=ws, stream=stream)

    def host(self):
        x = self.x
        inp = dict(q=x.q, k=x.k, v=x.v, g=x.g, beta=x.beta, dout=self.dout_h)
        if x.h0 is not None:
            inp["h0"] = x.h0
        self.h_in = {k: t.pin_memory() for k, t in inp.items()}
        s = self.s
        shapes = dict(dq=x.q.shape, dk=x.k.shape, dv=x.v.shape, dg=x.g.shape, dbeta=x.beta.shape,
                      dh0=(s["N"], s["Hv"], s["dk"], s["dv"]))
        self.h_out = [{k: self.torch.empty(sh, dtype=self.torch.float32).pin_memory() for k, sh in shapes.items()}
                      for _ in range(2)]
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * 4 for t in self.h_out[0].values()))

    def run(self, slot, ws, stream):
        self.step(slot, ws, stream)

    def d2h(self, slot):
        got = dict(zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), self.sets[slot]["grads"]))
        for k, t in self.h_out[slot].items():
            t.copy_(got[k], non_blocking=True)

    def config(self):
        c = super().config()
        c["pass"] = "backward, straight-through state QDQ"
        return c


class DecodeCase:
    """One step = one decode token for every (sequence, head); the state stays resident and is
    updated in place; the 64 token sets of the workload are cycled."""

    def __init__(self, d, dev, torch, gdn):
        self.d, self.dev, self.torch, self.gdn = d, dev, torch, gdn
        self.steps_avail = d.q.shape[0]
        self.tokens = d.q.shape[1]
        self.bytes = decode_bytes(d)
        _, N, Hqk, dk = d.q.shape
        Hv, dv = d.v.shape[2], d.v.shape[3]
        self.flops = N * Hv * 7 * dk * dv
        self.state = d.state.to(dev)
        self.tok = [dict(q=d.q[i].to(dev), k=d.k[i].to(dev), v=d.v[i].to(dev), g=d.g[i].to(dev),
                         beta=d.beta[i].to(dev)) for i in range(self.steps_avail)]
        self.o = torch.empty((N, Hv, dv), device=dev)
        self.launches = 1

    def workspace_bytes(self):
        return 0

    def scope(self):
        return "one step = one kernel launch"

    def step(self, i, ws, stream):
        t = self.tok[i % self.steps_avail]
        self.gdn.gdn_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], self.state, state_qdq=self.d.state_qdq,
                                 kda=self.d.kda, o=self.o, stream=stream, codec=self.d.codec)

    def host(self):
        self.h_in = {k: getattr(self.d, k)[0].pin_memory() for k in ("q", "k", "v", "g", "beta")}
        self.h_out = [self.torch.empty(self.o.shape, dtype=self.torch.float32).pin_memory() for _ in range(2)]
        self.o_slots = [self.o, self.torch.empty_like(self.o)]
        return sum(t.numel() * t.element_size() for t in self.h_in.values()), self.h_out[0].numel() * 4

    def h2d(self, slot):   # token inputs into the first two resident token sets
        for k, t in self.h_in.items():
            self.tok[slot][k].copy_(t, non_blocking=True)

    def run(self, slot, ws, stream):
        t = self.tok[slot]
        self.gdn.gdn_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], self.state, state_qdq=self.d.state_qdq,
                                 kda=self.d.kda, o=self.o_slots[slot], stream=stream, codec=self.d.codec)

    def d2h(self, slot):
        self.h_out[slot].copy_(self.o_slots[slot], non_blocking=True)

    def config(self):
        d = self.d
        return {"workload": d.name, "N": d.q.shape[1], "H": d.v.shape[2], "dk": d.q.shape[3], "dv": d.v.shape[3],
                "state_qdq": d.state_qdq, "codec": d.codec, "kda": d.kda,
                "state": "N(0,0.05), updated in place across steps"}


class QdqCase:
    """One step = one fp8_tile_qdq call over the whole tensor (out of place: x read, y and the
    tile scales written); two resident input sets alternate."""

    def __init__(self, d, dev, torch, gdn):
        self.d, self.dev, self.torch, self.gdn = d, dev, torch, gdn
        lead, rows, cols = d.x.shape
        ntiles = (cols + d.tile_cols - 1) // d.tile_cols
        self.tokens = lead * rows * cols                      # elements
        # E4M3: one scale per tile of a leading index; INT8: one per block of a row
        self.bytes = 8 * self.tokens + 4 * ntiles * (lead * rows if d.codec == "int8" else lead)
        self.flops = 0
        self.unit = "elements/s"
        self.xs = [d.x.to(dev), d.x.to(dev).neg_()]
        self.y = torch.empty_like(self.xs[0])
        self.launches = 1

    def workspace_bytes(self):
        return 0

    def scope(self):
        return "one step = one kernel launch"

    def _call(self, x, y, stream):
        if self.d.codec == "int8":
            self.gdn.int8_block_qdq(x, self.d.tile_cols, y=y, stream=stream)
        else:
            self.gdn.fp8_tile_qdq(x, self.d.tile_cols, y=y, stream=stream)

    def step(self, i, ws, stream):
        self._call(self.xs[i & 1], self.y, stream)

    def host(self):
        self.h_in = self.d.x.pin_memory()
        self.h_out = [self.torch.empty(self.y.shape, dtype=self.torch.float32).pin_memory() for _ in range(2)]
        self.y_slots = [self.y, self.torch.empty_like(self.y)]
        return self.h_in.numel() * 4, self.h_out[0].numel() * 4

    def h2d(self, slot):
        self.xs[slot].copy_(self.h_in, non_blocking=True)

    def run(self, slot, ws, stream):
        self._call(self.xs[slot], self.y_slots[slot], stream)

    def d2h(self, slot):
        self.h_out[slot].copy_(self.y_slots[slot], non_blocking=True)

    def config(self):
        d = self.d
        lead, rows, cols = d.x.shape
        c = {"workload": d.name, "lead": lead, "rows": rows, "cols": cols, "codec": d.codec,
             "x": "N(0,0.05) fp32, out of place"}
        c["block_cols" if d.codec == "int8" else "tile_cols"] = d.tile_cols
        return c


METRICS = {
    "gdn_b4_h16_t4096_d128": METRIC,
    "gdn_varlen8_hqk16_hv32_d128": "GDN varlen chunked-prefill tokens/s (8 seqs U[1,8192], GQA 16/32, d128, FP8 state QDQ)",
    "kda_b2_h32_t8192_d128": "KDA chunked-prefill tokens/s (B2 H32 T8192 d128, FP8 state + W QDQ)",
    "gdn_decode_n512_h32_d128_s64": "GDN decode tokens/s (N512 H32 d128, per-token FP8 state QDQ)",
    "qdq_state_n512_h32_d128": "standalone FP8 tile QDQ elements/s (16384 x [128 x 128] fp32, 64-column tiles)",
    "int8_state_n512_h32_d128": "standalone INT8 block QDQ elements/s (16384 x [128 x 128] fp32, 32-column blocks)",
    "gdn_bwd_b4_h16_t4096_d128": "GDN backward tokens/s (B4 H16 T4096 d128, straight-through FP8 state QDQ)",
    "kda_bwd_b2_h32_t8192_d128": "KDA backward tokens/s (B2 H32 T8192 d128, straight-through FP8 state QDQ)",
    "gdn_decode_int8_n512_h32_d128_s64": "GDN decode tokens/s (N512 H32 d128, per-token INT8 block-32 state QDQ)",
    "gdn_b1_h2_t256_d64": "GDN chunked-prefill tokens/s (B1 H2 T256 d64, FP8 state QDQ)",
    "handoff_n256_t128_p64_h16_d128": "GDN prefill->decode handoff tokens/s (256 seqs x 128 tokens, 64-token "
                                      "chunked prefix + 64 decode tokens, H16 d128, FP8 state + W QDQ)",
}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import fp8_state_qat_gb300 as gdn
    from fp8_state_qat_gb300 import workloads

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    gdn.load()
    dev = torch.device("cuda", local)
    x = workloads.workload(args.workload)
    if args.batch:   # profiling case of the same kernel: the first `batch` sequences
        x = workloads.PrefillInputs(x.q[:args.batch], x.k[:args.batch], x.v[:args.batch], x.g[:args.batch],
                                    x.beta[:args.batch], None if x.h0 is None else x.h0[:args.batch], None,
                                    kda=x.kda, state_qdq=x.state_qdq, w_qdq=x.w_qdq, name=x.name,
                                    backward=x.backward)
    if isinstance(x, workloads.DecodeInputs):
        case = DecodeCase(x, dev, torch, gdn)
    elif isinstance(x, workloads.QdqInputs):
        case = QdqCase(x, dev, torch, gdn)
    elif x.backward:
        case = BwdCase(x, dev, torch, gdn)
    else:
        case = PrefillCase(x, dev, torch, gdn)
    ws = torch.empty(max(case.workspace_bytes(), 1 << 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        case.step(i, ws, stream)
    torch.cuda.synchronize()
    gdn.gdn_check_device_status(ws)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        case.step(i, ws, stream)
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    if world > 1:
        dist.barrier()
    time.sleep(0.2)
    clocks.stop()
    gdn.gdn_check_device_status(ws)
    ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # end to end through the public API: every step copies its inputs from pinned host memory,
    # calls the library and copies its result back to pinned host memory. Copies in, calls and
    # copies out run on three streams with two buffer slots, so step i's call overlaps step i+1's
    # input copy and step i-1's output copy (the order a serving or training loop uses).
    h2d, d2h = case.host()
    e2e_steps = max(1, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_pipeline(steps):
        for i in range(steps):
            slot = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_run[slot])        # step i-2's call has read this slot's inputs
                case.h2d(slot)
                ev_in[slot].record(s_in)
            stream.wait_event(ev_in[slot])
            if i >= 2:
                stream.wait_event(ev_out[slot])          # step i-2's outputs have left this slot
            case.run(slot, ws, stream)
            ev_run[slot].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[slot])
                case.d2h(slot)
                ev_out[slot].record(s_out)

    e2e_pipeline(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_event(e0)
    s_out.wait_event(e0)
    e2e_pipeline(e2e_steps)
    s_out.wait_event(ev_run[(e2e_steps - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    if rank == 0:
        hbm, bf16, src = peaks()
        achieved = case.bytes / (launch_ms * 1e-3) / 1e9
        cfg = case.config()
        cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
        cfg["l2"] = "inputs larger than L2 (129 MB); prefill alternates two resident input sets"
        unit = getattr(case, "unit", UNIT)
        line = {"metric": METRICS.get(args.workload, args.workload), "value": job_rate(case.tokens * args.steps, world, ms),
                "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic", "config": cfg,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                             "frac": achieved / hbm,
                             "traffic": profiled_traffic(args.workload) if not args.batch else None,
                             "peak_source": src, "scope": case.scope(), "bytes_per_launch": case.bytes,
                             "flops_per_launch": case.flops,
                             "tensor_frac": case.flops / (launch_ms * 1e-3) / (bf16 * 1e12), "kernel_ms": launch_ms},
                "e2e": {"value": job_rate(case.tokens * e2e_steps, world, e2e_ms), "unit": unit,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
                "gpu_launches": args.steps * case.launches,
                "clocks": clocks.summary()}
        if getattr(case, "bound", "hbm") == "alu":
            clk = line["clocks"].get("sm_max_mhz") if isinstance(line["clocks"], dict) else None
            peak, psrc = alu_peak(dev, torch, clk)
            r = line["roofline"]
            tflops = case.flops / (launch_ms * 1e-3) / 1e12
            r.update({"bound": "alu", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                      "peak_source": psrc, "hbm_achieved_gbs": achieved, "hbm_frac": achieved / hbm})
        if world == 1 and not args.no_cpu_baseline and isinstance(case, PrefillCase) and args.workload == WORKLOAD:
            line["cpu_baseline"] = cpu_baseline(x)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(METRICS),
                    help="the benchmark is the default; the others measure the remaining hot-path rows")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling only: keep the first B sequences (the line is then not the benchmark)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
