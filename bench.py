#!/usr/bin/env python3
"""Benchmark: tokens/s and ms per gdr_chunk_fwd call on one GB300, with the
roofline fraction of the dominant kernel.

One step is one gdr_chunk_fwd call (the whole forward path: chunk indexing,
gate cumsum, Gram / inverse / WY factors, state scan, output, and for a long
sequence the segment pre-scan and composition) over one batch of the
headline workload, inputs resident in HBM: the largest configuration that
fits one GPU, one 65,536-token sequence with 8 heads (K = V = 128, BF16
q/k/v, near non-contracting decay), at the plan's segment count.  L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.

The same JSON line carries a sub-record per configuration ("configs"): ms
per call, tokens/s, the call's roofline fraction, per-kernel times; serial
beside split at 64K tokens (8 heads and 1); at 16K tokens every split count
with its error against the FP64 oracle on sampled (sequence, head) pairs;
the plan's pick beside serial on a batch with one long sequence; and the
backward pass (gdr_chunk_bwd, at its plan's route) on the wide varlen batch,
16K tokens and 64K tokens x 8 heads ("backward_<workload>").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdr|reference]
                  [--workload NAME] [--no-configs]

--impl reference times the FP64 CPU oracle (the slow reference program) on
bounded samples of the same workload, drawn by the same sampler as the
cpu_baseline record.  Under torchrun every rank runs an independent replica
(the path needs no exchange between GPUs); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/s and ms per gdr_chunk_fwd call on 1 GB300; % of roofline"
METRIC_BWD = "tokens/s and ms per gdr_chunk_bwd call on 1 GB300; % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "stress_64k_h8_bf16"
DEFAULT_WORKLOAD_BWD = "wide_varlen_bf16"  # the backward's headline: the wide varlen batch
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gdr", "reference"], default="gdr")
    ap.add_argument("--workload", default=None,
                    help=f"default {DEFAULT_WORKLOAD} ({DEFAULT_WORKLOAD_BWD} with --pass bwd)")
    ap.add_argument("--segments", type=int, default=0)
    ap.add_argument("--force-path", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sub-records")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd",
                    help="bwd times gdr_chunk_bwd (the backward pass) instead")
    args = ap.parse_args()
    if args.workload is None:
        args.workload = DEFAULT_WORKLOAD_BWD if args.which == "bwd" else DEFAULT_WORKLOAD
    return args


# ----------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ----------------------------------------------------------------------------
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK_PEAKS)
    p["source"] = "fallback"
    return p


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.gpu_index is not None:
                cmd += ["-i", str(self.gpu_index)]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


def gpu_index_for_smi():
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return local


# ----------------------------------------------------------------------------
# algorithmic bytes per kernel launch (units: token-heads, chunk-heads,
# sequence-heads, segment summaries)
# ----------------------------------------------------------------------------
def counts(x, n_segments=1, common=False):
    """Units of one call.  common: one segment length for every sequence,
    ceil(longest / S) chunks (the tensor-core delta forward), a sequence no
    longer than it left whole; else ceil(own chunks / S) per sequence."""
    H = x["H"]
    if x["cu_seqlens"] is not None:
        lens = (x["cu_seqlens"][1:] - x["cu_seqlens"][:-1]).tolist()
    else:
        lens = [x["T"]] * x["B"]
    chunks = sum((L + 63) // 64 for L in lens)
    segs = groups = split_tokens = split_chunks = split_seqs = 0
    S = max(1, n_segments)
    G = 0 if S < 4 else int(S ** 0.5)  # the two-level composition's group size
    longest = max([(L + 63) // 64 for L in lens] + [0])
    for L in lens:  # runs of whole chunks per sequence
        nc = (L + 63) // 64
        if common:
            per = -(-longest // S)
            ns = 0 if S == 1 or nc <= per else -(-nc // per)
        else:
            per = -(-nc // S) if nc else 0
            ns = -(-nc // per) if per else 0
        segs += ns
        groups += -(-ns // G) if G else 0
        if ns:
            split_tokens += L
            split_chunks += nc
            split_seqs += 1
    return dict(tokens=sum(lens), token_heads=sum(lens) * H, chunk_heads=chunks * H,
                seq_heads=len(lens) * H, n_seqs=len(lens), chunks=chunks, segments=segs * H,
                groups=groups * H, split_token_heads=split_tokens * H,
                split_chunk_heads=split_chunks * H, split_seq_heads=split_seqs * H)


def common_segments(x, plan):
    """The plan cuts sequences at one common segment length (the tensor-core
    forward, either mode)."""
    return plan.get("path") == 2


REC_BYTES = 57616  # bytes of one record written by tc_prep and read by the scan (k aside)


def algorithmic_bytes(kernel, x, c):
    K, V = x["K"], x["V"]
    es = 2 if x["dtype"] == "bf16" else 4
    delta = x["beta"] is not None
    th, ch, sh = c["token_heads"], c["chunk_heads"], c["seq_heads"]
    states = sh * K * V * 4 * ((1 if x["h0"] is not None else 0) + 1)
    # h0 / ht of the sequences a split composes (all of them but the empty
    # ones under each sequence's own run length; the split ones under a
    # common length, whose output pass takes the others whole)
    cstates = c["split_seq_heads"] * K * V * 4 * ((1 if x["h0"] is not None else 0) + 1)
    if kernel in ("call", "tc_gla_serial"):
        # whole forward pass: q, k, v, g, beta read once, o written once,
        # h0 / ht once
        return th * ((2 * K + V) * es + 4 + (4 if delta else 0) + V * es) + states
    if kernel == "tc_chain_serial":  # the records and k read, o written, states
        return th * (K + V) * es + ch * REC_BYTES + states
    if kernel == "tc_gla_prescan":  # k, v, g of the split sequences read; c_s written
        return c["split_token_heads"] * ((K + V) * es + 4) + c["segments"] * K * V * 4
    if kernel == "tc_gla_segment_out":  # q, k, v, g read, o written, h_s read
        return th * ((2 * K + V) * es + 4 + V * es) + c["segments"] * K * V * 4
    if kernel == "compose_scalar":  # c_s, d_s read; h_s written; h0 / ht
        return c["segments"] * (2 * K * V * 4 + 4) + cstates
    if kernel in ("compose_delta", "tc_compose"):  # M_s, c_s read; h_s written; h0 / ht
        return c["segments"] * ((K * K if delta else 1) + 2 * K * V) * 4 + cstates
    if kernel == "tc_compose_groups":  # M_s, c_s read; a group's transition and offset written
        return c["segments"] * (K * K + K * V) * 4 + c["groups"] * (K * K + K * V) * 4
    if kernel == "tc_compose_top":  # group transitions and offsets read; group states, h0 / ht
        return c["groups"] * (K * K + 2 * K * V) * 4 + cstates
    if kernel == "tc_compose_fill":  # M_s, c_s read; h_s written
        return c["segments"] * (K * K + 2 * K * V) * 4
    rec = ch * REC_BYTES  # per-chunk records of the tensor-core prep kernel
    if kernel == "tc_prep":  # q, k, v, g, beta read; records written
        return th * ((2 * K + V) * es + 8) + rec
    if kernel in ("tc_chain_prescan", "tc_prescan_dual"):
        # W, U^T, decay of the split sequences' records and k (once); c_s, M_s
        return (c["split_token_heads"] * K * es + c["split_chunk_heads"] * (2 * 16384 + 272)
                + c["segments"] * K * (K + V) * 4)
    if kernel == "tc_chain_segment_out":  # records and k read, o written, h_s read
        return th * (K + V) * es + rec + c["segments"] * K * V * 4
    if kernel == "simt_prep":
        b = th * 4 + ch * 64 * 4
        if delta:
            b += th * ((K + V) * es + 4) + ch * 64 * (K + V) * 4
        return b
    if kernel in ("simt_scan_serial", "simt_scan_segment_out"):
        b = th * K * es + ch * 64 * 4 + ch * K * V * 4
        b += (ch * 64 * (K + V) * 4 + ch * 64 * V * 4) if delta else th * V * es
        return b + (states if kernel == "simt_scan_serial" else sh * K * V * 4)
    if kernel == "simt_output":
        return (th * 2 * K * es + ch * K * V * 4 + ch * 64 * 4 + th * V * es
                + (ch * 64 * V * 4 if delta else th * V * es))
    return None


def bwd_algorithmic(kernel, x, c):
    """(bytes, flops) per launch of a backward-pass kernel (and of the forward
    recompute it runs): the operands each must read and the results it must
    write once, and the multiply-adds of the chunked form's products with
    causal halves counted once (L = 64 rows a chunk)."""
    K, V, L = x["K"], x["V"], 64
    es = 2 if x["dtype"] == "bf16" else 4
    delta = x["beta"] is not None
    th, ch, sh = c["token_heads"], c["chunk_heads"], c["seq_heads"]
    st = sh * K * V * 4
    f32 = 4
    if kernel == "bwd_gram":
        b = th * (2 * K * es + (4 if delta else 0)) + ch * L * f32 + ch * L * L * f32 * (3 if delta else 1)
        fma = ch * (L * L * K * (1.0 if delta else 0.5) + (L ** 3 / 6 if delta else 0))
    elif kernel == "bwd_dscan":
        b = (ch * L * L * f32 + th * (V + 2 * K) * es + ch * L * f32 + ch * K * V * f32
             + (ch * L * K * f32 + ch * L * V * f32 if delta else th * V * es) + 2 * st)
        fma = ch * (L * L * V / 2 + (3 if delta else 2) * L * K * V)
    elif kernel == "bwd_lk":
        b = (th * V * es + (2 * ch * L * V * f32 if delta else th * V * es) + 2 * ch * K * V * f32
             + ch * L * K * f32 * (3 if delta else 2))
        fma = ch * ((3 if delta else 2) * L * K * V + K * V)
    elif kernel == "bwd_local":
        b = (ch * L * L * f32 * (3 if delta else 1) + th * (2 * K + 2 * V) * es
             + ch * L * K * f32 * (3 if delta else 2) + ch * L * f32
             + (2 * ch * L * V * f32 + th * 4 if delta else th * V * es)
             + th * ((2 * K + (V if delta else 0)) * es + 4 + (4 if delta else 0)))
        fma = ch * (L * L * V / 2 + L * L * K)
        if delta:
            fma += ch * (1.5 * L * L * V + 2.5 * L * L * K + L ** 3 / 2)
    elif kernel == "tc_prep":  # the forward's preparation, plus G and T for the backward
        return algorithmic_bytes(kernel, x, c) + ch * L * f32 + ch * L * L * f32, None
    elif kernel == "tc_chain_recompute":
        # W^T, U^T, vectors, k read; v_new (FP32) and the BF16 image of the
        # h mirror written
        return (ch * (2 * 16384 + 272) + th * K * es + ch * L * V * f32 + ch * K * V * 2,
                None)
    elif kernel == "tc_chain_segment_recompute":  # as the serial recompute, from the segment states
        return (ch * (2 * 16384 + 272) + th * K * es + ch * L * V * f32 + ch * K * V * 2
                + c["segments"] * K * V * f32, None)
    elif kernel == "tc_bwd_scan":
        # W^T, Q~, P, vectors, k, dO read; dV' (a BF16 hi + lo pair) and the
        # BF16 image of the E mirror written; dht / dh0
        return (ch * (2 * 16384 + 8192 + 272) + th * (K + V) * es + ch * L * V * f32
                + ch * K * V * 2 + 2 * st, None)
    elif kernel == "tc_bwd_scan_prescan":  # the same reads; each segment's offset written
        return (ch * (2 * 16384 + 8192 + 272) + th * (K + V) * es
                + c["segments"] * K * V * f32, None)
    elif kernel == "tc_bwd_scan_segment_out":  # the serial scan's bytes from the segment ends
        return (ch * (2 * 16384 + 8192 + 272) + th * (K + V) * es + ch * L * V * f32
                + ch * K * V * 2 + c["segments"] * K * V * f32, None)
    elif kernel == "tc_bwd_grad":
        # h and E images, dO, q, k, v, T, dV', v_new (the FP32 operands as
        # BF16 hi + lo pairs: as many bytes as FP32), G, beta read; dq, dk,
        # dv, dbeta, dg written.  Its products run on the tensor cores, well
        # below their peak: HBM-bound.
        return (ch * 2 * K * V * 2 + th * (2 * V + 2 * K) * es + ch * L * L * f32
                + 2 * ch * L * V * f32 + ch * L * f32 + th * f32
                + th * (2 * K + V) * es + 2 * th * f32, None)
    elif kernel == "simt_prep":
        b = algorithmic_bytes(kernel, x, c)
        fma = ch * ((L * L * K / 2 + L ** 3 / 6 + L * L * (K + V) / 2) if delta else 0)
    elif kernel == "simt_scan_serial":
        b = algorithmic_bytes(kernel, x, c)
        fma = ch * (2 if delta else 1) * L * K * V
    else:
        return None, None
    return b, 2.0 * fma


# The translation unit each kernel is compiled from (plus every shared header).
KERNEL_SOURCES = {"tc_prep": "tc_prep.cu", "tc_chain": "tc_chain.cu", "tc_gla": "tc_gla.cu",
                  "tc_compose": "tc_compose.cu",
                  "tc_prescan": "tc_prescan.cu", "tc_bwd_scan": "tc_bwd_scan.cu",
                  "tc_bwd_grad": "tc_bwd_grad.cu", "recurrent": "recurrent.cu",
                  "compose": "compose.cu", "simt": "simt_path.cu", "bwd": "simt_bwd.cu"}


def traffic_record(kernel, workload):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = source_hash(kernel)
    for line in open(path):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if (f.get("kernel") == kernel and f.get("workload") == workload
                and f.get("source_sha") == src):
            return float(f["dram_bytes_per_launch"])
    return None


def kernel_sources(kernel):
    """The kernel's .cu file and every package header it includes, directly
    or through other headers (file names, the .cu file first)."""
    import re
    csrc = os.path.join(ROOT, "chunked_gated_delta_rule_gb300", "csrc")
    main = next((v for k, v in KERNEL_SOURCES.items() if kernel.startswith(k)), None)
    if main is None:
        main = "compose.cu" if "compose" in kernel else "simt_path.cu"
    seen, order, todo = set(), [], [main]
    while todo:
        f = todo.pop(0)
        if f in seen or not os.path.exists(os.path.join(csrc, f)):
            continue
        seen.add(f)
        order.append(f)
        todo += re.findall(r'#include\s+"([^"]+)"', open(os.path.join(csrc, f)).read())
    return [order[0]] + sorted(order[1:])


def source_hash(kernel):
    """sha256 (16 hex digits) of kernel_sources(kernel)."""
    csrc = os.path.join(ROOT, "chunked_gated_delta_rule_gb300", "csrc")
    h = hashlib.sha256()
    for f in kernel_sources(kernel):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------
# CPU oracle timing (reported baseline / reference arm).  One sampler serves
# both: a sample is whole heads of a few sequences taken in order (cycling),
# each cut to its first ORACLE_SAMPLE_TOKENS tokens, until that many tokens
# are taken; the oracle's cost per token does not depend on the position.
# ----------------------------------------------------------------------------
ORACLE_SAMPLE_TOKENS = 4096


def oracle_sample(x, first, cap=ORACLE_SAMPLE_TOKENS):
    """Rows of one sample: a list of (sequence, first row, rows) along the
    flattened token axis, starting at sequence `first`; returns (pieces,
    tokens, next sequence)."""
    if x["cu_seqlens"] is not None:
        cu = [int(c) for c in x["cu_seqlens"].tolist()]
    else:
        cu = [n * x["T"] for n in range(x["B"] + 1)]
    N = len(cu) - 1
    pieces, tokens, n, seen = [], 0, first % N, 0
    while tokens < cap and seen < N:
        a, b = cu[n], cu[n + 1]
        take = min(b - a, cap - tokens)
        if take > 0:
            pieces.append((n, a, take))
            tokens += take
        n = (n + 1) % N
        seen += 1
    return pieces, tokens, n


def sample_inputs(xo, pieces, extra=None):
    """The sample as its own varlen problem (FP64 arrays, all heads):
    q, k, v, g, beta, h0 and the optional per-token / per-sequence extras
    (do, dht) cut to the sample's rows and sequences."""
    import numpy as np

    def rows(a):
        if a is None:
            return None
        flat = a.reshape((-1,) + a.shape[2:])
        return np.ascontiguousarray(np.concatenate([flat[r:r + n] for _, r, n in pieces])[None])

    def seqs(a):
        return None if a is None else np.ascontiguousarray(a[[s for s, _, _ in pieces]])

    cu = np.zeros(len(pieces) + 1, dtype=np.int64)
    cu[1:] = np.cumsum([n for _, _, n in pieces])
    sub = {k: rows(xo[k]) for k in ("q", "k", "v", "g", "beta")}
    sub.update(cu_seqlens=cu, h0=seqs(xo["h0"]), H=xo["H"])
    if extra:
        sub["do"] = rows(extra[0])
        sub["dht"] = seqs(extra[1])
    return sub


def oracle_inputs(x):
    import oracle
    return {k: (oracle._f64(v) if k in ("q", "k", "v", "g", "beta", "h0") else v)
            for k, v in x.items()}


def time_oracle_sample(sub, backward=False):
    """Seconds and threads of one oracle run on a sample (all heads)."""
    import oracle
    t0 = time.perf_counter()
    if backward:
        oracle.backward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                        cu_seqlens=sub["cu_seqlens"], h0=sub["h0"], do=sub["do"], dht=sub["dht"])
        threads = min(os.cpu_count() or 1, (len(sub["cu_seqlens"]) - 1) * sub["H"])
    else:
        _, _, threads = oracle.forward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                       cu_seqlens=sub["cu_seqlens"], h0=sub["h0"], want_ht=True)
    return time.perf_counter() - t0, threads


def bwd_grads_in(x, seed=7):
    """Seeded incoming gradients of the backward benchmark: do in the input
    dtype, dht FP32."""
    import torch
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype)
    dht = torch.randn(x["N"], x["H"], x["K"], x["V"], generator=gen)
    return do, dht


def oracle_samples(x, backward=False):
    """Generator of (seconds, tokens, threads) over successive samples of
    the workload; the first untimed run loads the oracle."""
    import oracle
    xo = oracle_inputs(x)
    extra = None
    if backward:
        do, dht = bwd_grads_in(x)
        extra = (oracle._f64(do), oracle._f64(dht))
    nxt = 0
    pieces, _, _ = oracle_sample(x, 0, cap=64)
    time_oracle_sample(sample_inputs(xo, pieces, extra), backward)  # load, untimed
    while True:
        pieces, tokens, nxt = oracle_sample(x, nxt)
        secs, threads = time_oracle_sample(sample_inputs(xo, pieces, extra), backward)
        yield secs, tokens, threads, len(pieces)


def sample_text(x, backward):
    return (f"samples of up to {ORACLE_SAMPLE_TOKENS} tokens: whole heads ({x['H']}) of "
            f"sequences taken in order, each cut to its first {ORACLE_SAMPLE_TOKENS} tokens; "
            "FP64 token recurrence" + (" and its reverse (backward)" if backward else ""))


def cpu_baseline(x, budget_s, backward=False):
    """The oracle on successive samples until about `budget_s` seconds of
    CPU work."""
    secs = toks = n = 0
    threads = 1
    for dt, tk, threads, _ in oracle_samples(x, backward):
        secs += dt
        toks += tk
        n += 1
        if secs >= budget_s or n >= 256:
            break
    return {"value": toks / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} {sample_text(x, backward)}; {toks} tokens in {secs:.1f} s"}


def cpu_baseline_bwd(x, budget_s):
    return cpu_baseline(x, budget_s, backward=True)


def run_reference(args):
    from chunked_gated_delta_rule_gb300 import synthetic
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synthetic.WORKLOADS[args.workload]
    x = synthetic.make_inputs(w)
    backward = args.which == "bwd"
    times, toks, threads = [], [], 1
    gen = oracle_samples(x, backward)
    for i in range(args.warmup + args.steps):
        dt, tk, threads, _ = next(gen)
        if i >= args.warmup:
            times.append(dt)
            toks.append(tk)
    value = sum(toks) / sum(times)
    line = {"impl": "reference", "metric": METRIC_BWD if backward else METRIC,
            "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, x, None),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "each step one of the " + sample_text(x, backward)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def config_of(args, x, plan):
    c = {"workload": args.workload, "tokens": None, "n_seqs": x["N"], "H": x["H"],
         "K": x["K"], "V": x["V"], "input_dtype": x["dtype"],
         "beta_free": x["beta"] is None, "h0": x["h0"] is not None,
         "l2": "flushed between timed steps (256 MiB write, untimed)"}
    c["tokens"] = counts(x)["tokens"]
    if plan is not None:
        c["plan"] = plan
    return c


def scan_bytes(x, c):
    """Algorithmic bytes of the state scan alone (its unfused form, the BF16
    state stored once a chunk), per the hot-path table: per token-head W and
    U (delta rule), k, g, v_new, and K*V*2/64 of state; 1,540 B at K = V =
    128 BF16."""
    K, V = x["K"], x["V"]
    es = 2 if x["dtype"] == "bf16" else 4
    delta = x["beta"] is not None
    per = ((K + V) * es if delta else 0) + K * es + 4 + V * es + K * V * 2 / 64
    return c["token_heads"] * per


def max_seqlen_of(x):
    if x["cu_seqlens"] is None:
        return None
    cu = x["cu_seqlens"]
    return int((cu[1:] - cu[:-1]).max()) if cu.numel() > 1 else 0


def plan_of(pkg, x, segments=0):
    return pkg.gdr_plan_query(x["B"], x["T"], x["H"], x["K"], x["V"],
                              N=x["N"] if x["cu_seqlens"] is not None else 0,
                              dtype={"f32": 0, "bf16": 1, "f16": 2}[x["dtype"]],
                              beta_free=x["beta"] is None, n_segments=segments,
                              max_len=max_seqlen_of(x) or 0)


class Measured:
    """Timed gdr_chunk_fwd calls on one workload: `steps` calls bracketed by
    CUDA events on the launching stream with L2 flushed between them, then a
    second pass of the same calls with the library's per-launch events."""

    def __init__(self, pkg, x, dev, steps, warmup, flush, n_segments=0, force_path=0,
                 sampler=None, kernels=True):
        import torch
        self.x = x
        d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
        self.d = d
        o = torch.empty_like(d["v"])
        ht = torch.empty(x["N"], x["H"], x["K"], x["V"], dtype=torch.float32, device=dev)
        self.kw = dict(cu_seqlens=d["cu_seqlens"], h0=d["h0"], o=o, ht=ht,
                       n_segments=n_segments, force_path=force_path,
                       max_seqlen=max_seqlen_of(x))
        self.args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
        stream = torch.cuda.current_stream(dev)
        for _ in range(max(3, warmup)):
            pkg.gdr_chunk_fwd(*self.args, **self.kw)
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        if sampler:
            sampler.start()
            time.sleep(0.3)
        # A bounded ~2 ms spin on the GPU and one untimed call behind it,
        # outside the timed region, so that the host is already enqueueing
        # the steps when the first one starts.
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(4_000_000)
        pkg.gdr_chunk_fwd(*self.args, **self.kw)
        for i in range(steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            pkg.gdr_chunk_fwd(*self.args, **self.kw)
            ends[i].record(stream)
        torch.cuda.synchronize()
        self.clocks = sampler.stop() if sampler else None
        self.step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        self.ms = statistics.mean(self.step_ms)
        self.per_kernel, self.launches, self.kstep_ms = {}, 0, []
        if not kernels:
            return
        timers = [pkg.LaunchTimer(16) for _ in range(steps)]
        ks = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ke = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ks[i].record(stream)
            pkg.gdr_chunk_fwd(*self.args, timer=timers[i], **self.kw)
            ke[i].record(stream)
        torch.cuda.synchronize()
        self.kstep_ms = [a.elapsed_time(b) for a, b in zip(ks, ke)]
        for t in timers:
            self.launches += t.count
            for i, kid in enumerate(t.ids):
                self.per_kernel.setdefault(pkg.gdr_kernel_name(kid), []).append(t.elapsed_ms(i))

    def kernels(self):
        tot = sum(self.kstep_ms) or 1.0
        return {n: {"launches": len(v), "avg_ms": statistics.mean(v), "share": sum(v) / tot}
                for n, v in self.per_kernel.items()}

    def outputs(self):
        return self.kw["o"], self.kw["ht"]


def rooflines(x, c, m, hbm, workload):
    """Fractions of the measured copy bandwidth, by the hot-path table's
    algorithmic bytes: the whole call's 1,032 B per token-head (K = V = 128
    BF16) over the dominant kernel's mean launch time (`roofline`) and over
    the call (`call_roofline`); the scan alone's 1,540 B per token-head over
    the scan kernel's time (`scan_roofline`).  Each kernel's own bytes
    (its records and summaries included) go under kernel_bytes."""
    call = algorithmic_bytes("call", x, c)
    out = {"call_roofline": {"achieved": call / (m.ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": call / (m.ms * 1e-3) / 1e9 / hbm, "algorithmic_bytes": call}}
    if not m.per_kernel:
        return out
    dom = max(m.per_kernel, key=lambda n: sum(m.per_kernel[n]))
    dom_ms = statistics.mean(m.per_kernel[dom])
    own = algorithmic_bytes(dom, x, c)
    out["roofline"] = {
        "kernel": dom, "bound": "hbm", "achieved": call / (dom_ms * 1e-3) / 1e9, "peak": hbm,
        "unit": "GB/s", "frac": call / (dom_ms * 1e-3) / 1e9 / hbm,
        "traffic": traffic_record(dom, workload),
        "algorithmic_bytes_per_launch": call, "avg_launch_ms": dom_ms,
        "kernel_bytes": own,
        "kernel_frac": own / (dom_ms * 1e-3) / 1e9 / hbm if own else None,
        "basis": "the whole call's algorithmic bytes (q, k, v, g, beta read once, o written "
                 "once, h0 / ht) over the dominant kernel's mean launch time; kernel_bytes "
                 "is the kernel's own traffic, per-chunk records included"}
    scan = next((n for n in ("tc_chain_serial", "tc_chain_segment_out", "tc_gla_serial",
                             "tc_gla_segment_out", "simt_scan_serial", "simt_scan_segment_out")
                 if n in m.per_kernel), None)
    if scan is not None:
        sb = scan_bytes(x, c)
        s_ms = statistics.mean(m.per_kernel[scan])
        own = algorithmic_bytes(scan, x, c)
        out["scan_roofline"] = {
            "kernel": scan, "bound": "hbm", "achieved": sb / (s_ms * 1e-3) / 1e9, "peak": hbm,
            "unit": "GB/s", "frac": sb / (s_ms * 1e-3) / 1e9 / hbm,
            "traffic": traffic_record(scan, workload), "algorithmic_bytes_per_launch": sb,
            "avg_launch_ms": s_ms, "kernel_bytes": own,
            "kernel_frac": own / (s_ms * 1e-3) / 1e9 / hbm if own else None}
    return out


# Per-configuration sub-records: the five configurations of the project
# statement (64K at 8 and 1 heads) and a batch with one long sequence.
CONFIG_WORKLOADS = ("tiny_dense_f32", "wide_varlen_bf16", "long_16k_bf16", "stress_64k_h8_bf16",
                    "stress_64k_h1_bf16", "gla_k256_v512_bf16", "skewed_varlen_bf16",
                    "skewed_varlen_h4_bf16", "skewed_gla_h4_bf16")


def config_record(pkg, name, dev, steps, flush, hbm):
    from chunked_gated_delta_rule_gb300 import synthetic
    x = synthetic.make_inputs(synthetic.WORKLOADS[name])
    plan = plan_of(pkg, x)
    c = counts(x, plan["n_segments"], common_segments(x, plan))
    m = Measured(pkg, x, dev, steps, 3, flush)
    rec = {"plan": plan, "tokens": c["tokens"], "ms_per_call": m.ms,
           "tokens_per_s": c["tokens"] / (m.ms * 1e-3),
           "token_heads_per_s": c["token_heads"] / (m.ms * 1e-3),
           "kernels": m.kernels()}
    rec.update(rooflines(x, c, m, hbm, name))
    if name.startswith("skewed"):
        ser = Measured(pkg, x, dev, steps, 3, flush, n_segments=1, kernels=False)
        rec["serial_ms_per_call"] = ser.ms
        rec["split_over_serial_speedup"] = ser.ms / m.ms
        del ser
    if name in SPLIT_SWEEPS:
        add_split_sweep(rec, pkg, x, dev, steps, flush, plan["n_segments"], SPLIT_SWEEPS[name])
    return x, m, rec


# Backward sub-records of the default line: gdr_chunk_bwd at its plan's
# route, do / dht seeded, L2 flushed between timed calls.
BWD_CONFIG_WORKLOADS = ("wide_varlen_bf16", "long_16k_bf16", "stress_64k_h8_bf16")


def bwd_config_record(pkg, name, dev, steps, flush):
    import torch
    from chunked_gated_delta_rule_gb300 import synthetic
    x = synthetic.make_inputs(synthetic.WORKLOADS[name])
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    do_h, dht_h = bwd_grads_in(x)
    do, dht = do_h.to(dev), dht_h.to(dev)
    args_t = (d["q"], d["k"], d["v"], d["g"], d["beta"], do)
    kw = dict(cu_seqlens=d["cu_seqlens"], h0=d["h0"], dht=dht)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        pkg.gdr_chunk_bwd(*args_t, **kw)
    ts, per = [], {}
    for i in range(2 * steps):
        flush.fill_(i & 0xFF)
        timer = pkg.LaunchTimer(16) if i % 2 else None
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkg.gdr_chunk_bwd(*args_t, timer=timer, **kw)
        e1.record(stream)
        torch.cuda.synchronize()
        if timer is None:
            ts.append(e0.elapsed_time(e1))
        else:
            for j, kid in enumerate(timer.ids):
                per.setdefault(pkg.gdr_kernel_name(kid), []).append(timer.elapsed_ms(j))
    ms = statistics.mean(ts)
    c = counts(x)
    kernels = {k: {"launches_per_call": len(v) // steps, "avg_ms": statistics.mean(v)}
               for k, v in per.items()}
    route = "tensor cores" if "tc_bwd_grad" in kernels else "CUDA cores (FP32)"
    rec = {"route": route, "tokens": c["tokens"], "ms_per_call": ms,
           "tokens_per_s": c["tokens"] / (ms * 1e-3), "kernels": kernels}
    del d, do, dht
    return rec


def add_split_sweep(rec, pkg, x, dev, steps, flush, plan_s, counts_):
    """ms per call at each split count and the error against the serial
    result on the same inputs (the pages' "CP vs serial" accuracy table;
    the errors against the FP64 oracle at each count are the GPU parity
    tests', on sampled pairs).  At strong decay (g ~ log sigmoid(N(3, 1)))
    a segment's transition underflows to zero in FP32 and the split is
    bit-identical to serial; the near non-contracting 64K workload is where
    split counts differ."""
    sweep = {}
    o1 = ht1 = None
    for S in sorted(set(counts_) | {plan_s, 1}):
        mS = Measured(pkg, x, dev, steps, 3, flush, n_segments=S, kernels=False)
        o, ht = mS.outputs()
        if S == 1:
            o1, ht1 = o.clone(), ht.clone()
        sweep[str(S)] = {"ms_per_call": mS.ms, "rel_l2_vs_serial_o": rel_l2(o, o1),
                         "rel_l2_vs_serial_ht": rel_l2(ht, ht1)}
        del mS, o, ht
    rec["split_sweep"] = sweep
    rec["serial_ms_per_call"] = sweep["1"]["ms_per_call"]
    rec["split_over_serial_speedup"] = sweep["1"]["ms_per_call"] / sweep[str(plan_s)]["ms_per_call"]


# split counts swept per configuration (the plan's count is always added)
# (128 segments of the beta-free batch: one chunk each, the chunk-parallel
# producer dataflow)
SPLIT_SWEEPS = {"long_16k_bf16": (1, 2, 4, 8, 16), "stress_64k_h8_bf16": (1, 4, 8, 16),
                "stress_64k_h1_bf16": (1, 16, 32, 64), "gla_k256_v512_bf16": (1, 4, 16, 128)}


def rel_l2(a, ref):
    """||a - ref|| / ||ref|| in FP64 on the device."""
    a64, r64 = a.double(), ref.double()
    den = float(r64.norm())
    return float((a64 - r64).norm()) / den if den > 0 else float((a64 - r64).norm())


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_gdr(args):
    import torch
    import chunked_gated_delta_rule_gb300 as pkg
    from chunked_gated_delta_rule_gb300 import synthetic

    rank, local, world = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synthetic.WORKLOADS[args.workload]
    x = synthetic.make_inputs(w)
    plan = plan_of(pkg, x, args.segments)
    seg_count = plan["n_segments"]
    if args.force_path and args.force_path != plan["path"]:
        # the query plans the default path; a forced path applies its own rules
        seg_count = args.segments or 1
        plan = {"path": args.force_path, "bv": "per the forced path's rule",
                "n_segments": args.segments or "per the forced path's rule"}
    c = counts(x, seg_count, common_segments(x, plan))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    hbm = float(peaks["hbm_gbs"])

    K = args.steps
    sampler = ClockSampler(gpu_index_for_smi()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    m = Measured(pkg, x, dev, K, args.warmup, flush, n_segments=args.segments,
                 force_path=args.force_path, sampler=sampler)
    barrier(world)
    clocks = m.clocks
    ms = max_over_ranks(m.ms, world)
    roof = rooflines(x, c, m, hbm, args.workload)
    roofline = roof.get("roofline")
    if roofline is not None:
        roofline["timing"] = ("CUDA events around each launch on its stream, over a second "
                              "pass of the same K steps")
        roofline["peak_source"] = peaks["source"] + " (hbm_gbs, copy bandwidth)"
    call_roofline = dict(roof["call_roofline"])
    call_roofline.update(achieved=roof["call_roofline"]["algorithmic_bytes"] / (ms * 1e-3) / 1e9,
                         frac=roof["call_roofline"]["algorithmic_bytes"] / (ms * 1e-3) / 1e9 / hbm)
    kernels = m.kernels()
    launches = m.launches
    step_ms = m.step_ms

    e2e = None
    if not args.no_e2e:
        pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
        o, ht = m.outputs()
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        ht_h = torch.empty(ht.shape, dtype=ht.dtype).pin_memory()
        hargs = (pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"])
        hkw = dict(cu_seqlens=pin["cu_seqlens"], h0=pin["h0"], o=o_h, ht=ht_h,
                   n_segments=args.segments)
        for _ in range(3):
            pkg.gdr_chunk_fwd_host(*hargs, **hkw)
        ke = max(3, min(K, 50))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ke):
            pkg.gdr_chunk_fwd_host(*hargs, **hkw)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / ke, world)
        h2d = sum(t.numel() * t.element_size() for t in
                  [pin[k] for k in ("q", "k", "v", "g", "beta", "cu_seqlens", "h0")]
                  if t is not None)
        d2h = o_h.numel() * o_h.element_size() + ht_h.numel() * ht_h.element_size()
        e2e = {"value": world * c["tokens"] / (e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": ke, "api": "gdr_chunk_fwd_host (pinned host buffers)"}
        del pin, o_h, ht_h

    configs = None
    if rank == 0 and not args.no_configs and not args.force_path and args.segments == 0:
        configs = {}
        del m
        torch.cuda.empty_cache()
        for name in CONFIG_WORKLOADS:
            if name == args.workload:
                configs[name] = {"plan": plan, "tokens": c["tokens"], "ms_per_call": ms,
                                 "tokens_per_s": c["tokens"] / (ms * 1e-3),
                                 "token_heads_per_s": c["token_heads"] / (ms * 1e-3),
                                 "kernels": kernels, **roof, "headline": True}
                if name in SPLIT_SWEEPS:
                    add_split_sweep(configs[name], pkg, x, dev, min(K, 20), flush,
                                    plan["n_segments"], SPLIT_SWEEPS[name])
                continue
            _, cm, rec = config_record(pkg, name, dev, min(K, 20), flush, hbm)
            configs[name] = rec
            del cm
            torch.cuda.empty_cache()
        for name in BWD_CONFIG_WORKLOADS:
            configs["backward_" + name] = bwd_config_record(pkg, name, dev, min(K, 10), flush)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": world * c["tokens"] / (ms * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None,
                "dtype": "f32" if plan["path"] == 1 else "bf16",
                "data": "synthetic (seeded; shapes and distributions of the workload)",
                "config": config_of(args, x, plan),
                "roofline": roofline, "scan_roofline": roof.get("scan_roofline"),
                "call_roofline": call_roofline,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "kernels": kernels, "clocks": clocks,
                "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                            "p10": sorted(step_ms)[len(step_ms) // 10],
                            "p90": sorted(step_ms)[(9 * len(step_ms)) // 10]},
                "configs": configs}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()




def run_decode(args):
    """gdr_recurrent_fwd on a decode workload: every sequence one token,
    continuing a state held at a seeded row of a pool twice the batch."""
    import torch
    import chunked_gated_delta_rule_gb300 as pkg
    from chunked_gated_delta_rule_gb300 import synthetic

    rank, local, world = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synthetic.WORKLOADS[args.workload]
    x = synthetic.make_inputs(w)
    pool_h, idx_h = synthetic.make_state_pool(x, 2 * x["N"])
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    pool, idx = pool_h.to(dev), idx_h.to(dev)
    o = torch.empty_like(d["v"])
    args_t = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    kw = dict(cu_seqlens=d["cu_seqlens"], state=pool, state_indices=idx, o=o)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        pkg.gdr_recurrent_fwd(*args_t, **kw)
    torch.cuda.synchronize()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_index_for_smi()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if hasattr(torch.cuda, "_sleep"):  # outside the timed region, as in run_gdr
        torch.cuda._sleep(4_000_000)
    pkg.gdr_recurrent_fwd(*args_t, **kw)
    for i in range(K):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        pkg.gdr_recurrent_fwd(*args_t, **kw)
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world)

    H, Kd, V = x["H"], x["K"], x["V"]
    es = 2 if x["dtype"] == "bf16" else 4
    tokens = int(x["cu_seqlens"][-1]) if x["cu_seqlens"] is not None else x["B"] * x["T"]
    ab = x["N"] * H * 2 * Kd * V * 4 + tokens * H * ((2 * Kd + V) * es + 8 + V * es)
    peaks = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = ab / (ms * 1e-3) / 1e9
    roofline = {"kernel": "recurrent", "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic_record("recurrent", args.workload),
                "algorithmic_bytes_per_launch": ab, "avg_launch_ms": ms,
                "timing": "CUDA events around each call (one kernel launch) on its stream",
                "peak_source": peaks["source"] + " (hbm_gbs, copy bandwidth)"}

    e2e = None
    if not args.no_e2e:
        pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        names = ("q", "k", "v", "g", "beta", "cu_seqlens")

        def e2e_step():
            for nme in names:
                if pin[nme] is not None:
                    d[nme].copy_(pin[nme], non_blocking=True)
            pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  cu_seqlens=d["cu_seqlens"], state=pool, state_indices=idx, o=o)
            o_h.copy_(o, non_blocking=True)

        for _ in range(3):
            e2e_step()
        ke = max(3, min(K, 50))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / ke, world)
        h2d = sum(pin[nme].numel() * pin[nme].element_size() for nme in names
                  if pin[nme] is not None)
        e2e = {"value": world * tokens / (e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": o_h.numel() * o_h.element_size(),
               "ms_per_step": e_ms, "steps": ke,
               "api": "gdr_recurrent_fwd, inputs and o through pinned host buffers, "
                      "the state pool resident on the device"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, args.cpu_seconds)
    if rank == 0:
        line = {"metric": METRIC, "value": world * tokens / (ms * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded; shapes and distributions of the workload)",
                "config": {"workload": args.workload, "tokens": tokens, "n_seqs": x["N"],
                           "H": H, "K": Kd, "V": V, "input_dtype": x["dtype"],
                           "beta_free": x["beta"] is None, "state_pool_rows": 2 * x["N"],
                           "l2": "flushed between timed steps (256 MiB write, untimed)",
                           "entry_point": "gdr_recurrent_fwd"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K,
                "clocks": clocks,
                "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                            "p10": sorted(step_ms)[len(step_ms) // 10],
                            "p90": sorted(step_ms)[(9 * len(step_ms)) // 10]}}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_bwd(args):
    """gdr_chunk_bwd on a workload: the gradients of <do, o> + <dht, ht> for
    seeded do / dht, inputs resident in HBM."""
    import torch
    import chunked_gated_delta_rule_gb300 as pkg
    from chunked_gated_delta_rule_gb300 import synthetic

    rank, local, world = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synthetic.WORKLOADS[args.workload]
    x = synthetic.make_inputs(w)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}
    do_h, dht_h = bwd_grads_in(x)
    do, dht = do_h.to(dev), dht_h.to(dev)
    outs = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]),
                dv=torch.empty_like(d["v"]), dg=torch.empty_like(d["g"]),
                dbeta=None if d["beta"] is None else torch.empty_like(d["beta"]),
                dh0=torch.empty(x["N"], x["H"], x["K"], x["V"], dtype=torch.float32, device=dev))
    args_t = (d["q"], d["k"], d["v"], d["g"], d["beta"], do)
    kw = dict(cu_seqlens=d["cu_seqlens"], h0=d["h0"], dht=dht, n_segments=args.segments,
              force_path=args.force_path, **outs)
    c = counts(x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        pkg.gdr_chunk_bwd(*args_t, **kw)
    torch.cuda.synchronize()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_index_for_smi()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if hasattr(torch.cuda, "_sleep"):  # outside the timed region, as in run_gdr
        torch.cuda._sleep(4_000_000)
    pkg.gdr_chunk_bwd(*args_t, **kw)
    for i in range(K):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        pkg.gdr_chunk_bwd(*args_t, **kw)
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world)

    timers = [pkg.LaunchTimer(16) for _ in range(K)]
    kstarts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    kends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        kstarts[i].record(stream)
        pkg.gdr_chunk_bwd(*args_t, timer=timers[i], **kw)
        kends[i].record(stream)
    torch.cuda.synchronize()
    kstep_ms = [s.elapsed_time(e) for s, e in zip(kstarts, kends)]
    per_kernel, launches = {}, 0
    for t in timers:
        launches += t.count
        for i, kid in enumerate(t.ids):
            per_kernel.setdefault(pkg.gdr_kernel_name(kid), []).append(t.elapsed_ms(i))
    kernels = {}
    peaks = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    sm_mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    fp32_tflops = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12
    for n, v in per_kernel.items():
        b, f = bwd_algorithmic(n, x, c)
        k_ms = statistics.mean(v)
        kernels[n] = {"launches": len(v), "avg_ms": k_ms, "share": sum(v) / sum(kstep_ms),
                      "hbm_frac": b / (k_ms * 1e-3) / 1e9 / hbm if b else None,
                      "fp32_frac": f / (k_ms * 1e-3) / 1e12 / fp32_tflops if f else None}
    dom = max(per_kernel, key=lambda n: sum(per_kernel[n]))
    b, f = bwd_algorithmic(dom, x, c)
    dom_ms = statistics.mean(per_kernel[dom])
    hb = b / (dom_ms * 1e-3) / 1e9 if b else 0.0
    fl = f / (dom_ms * 1e-3) / 1e12 if f else 0.0
    if f and fl / fp32_tflops >= hb / hbm:
        roofline = {"kernel": dom, "bound": "alu", "achieved": fl, "peak": fp32_tflops,
                    "unit": "TFLOP/s", "frac": fl / fp32_tflops,
                    "traffic": traffic_record(dom, "bwd_" + args.workload),
                    "algorithmic_flops_per_launch": f, "avg_launch_ms": dom_ms,
                    "peak_source": "FP32 CUDA-core peak: 152 SMs x 128 lanes x 2 flops x "
                                   f"{sm_mhz:.0f} MHz (no measured FP32 peak)"}
    else:
        roofline = {"kernel": dom, "bound": "hbm", "achieved": hb, "peak": hbm, "unit": "GB/s",
                    "frac": hb / hbm, "traffic": traffic_record(dom, "bwd_" + args.workload),
                    "algorithmic_bytes_per_launch": b, "avg_launch_ms": dom_ms,
                    "peak_source": peaks["source"] + " (hbm_gbs, copy bandwidth)"}
    roofline["timing"] = ("CUDA events around each launch on its stream, over a second pass "
                          "of the same K steps")
    es = 2 if x["dtype"] == "bf16" else 4
    th, Kd, V = c["token_heads"], x["K"], x["V"]
    delta = x["beta"] is not None
    call_bytes = (th * ((2 * Kd + 2 * V) * es + 4 + (4 if delta else 0))      # q k v do g beta
                  + th * ((2 * Kd + V) * es + 4 + (4 if delta else 0))        # dq dk dv dg dbeta
                  + c["seq_heads"] * Kd * V * 4 * (2 + (1 if x["h0"] is not None else 0)))
    call_roofline = {"achieved": call_bytes / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": call_bytes / (ms * 1e-3) / 1e9 / hbm, "algorithmic_bytes": call_bytes}

    e2e = None
    if not args.no_e2e:
        pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
        do_p, dht_p = do_h.pin_memory(), dht_h.pin_memory()
        host_out = {k: (None if v is None else torch.empty(v.shape, dtype=v.dtype).pin_memory())
                    for k, v in outs.items()}
        names = ("q", "k", "v", "g", "beta", "cu_seqlens", "h0")

        def e2e_step():
            for nme in names:
                if pin[nme] is not None:
                    d[nme].copy_(pin[nme], non_blocking=True)
            do.copy_(do_p, non_blocking=True)
            dht.copy_(dht_p, non_blocking=True)
            pkg.gdr_chunk_bwd(*args_t, **kw)
            for k2, t in outs.items():
                if t is not None:
                    host_out[k2].copy_(t, non_blocking=True)

        for _ in range(3):
            e2e_step()
        ke = max(3, min(K, 20))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / ke, world)
        h2d = sum(pin[nme].numel() * pin[nme].element_size() for nme in names
                  if pin[nme] is not None) + do_p.numel() * do_p.element_size() + dht_p.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in host_out.values() if t is not None)
        e2e = {"value": world * c["tokens"] / (e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": ke, "api": "gdr_chunk_bwd, inputs and gradients through pinned host "
                                   "buffers (copies on the calling stream)"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_bwd(x, args.cpu_seconds)
    if rank == 0:
        cfg = config_of(args, x, None)
        cfg["entry_point"] = "gdr_chunk_bwd"
        cfg["n_segments"] = args.segments or "auto"
        cfg["incoming_gradients"] = "do ~ N(0,1) in the input dtype, dht ~ N(0,1) FP32, seed 7"
        line = {"metric": METRIC_BWD, "value": world * c["tokens"] / (ms * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded; shapes and distributions of the workload)",
                "config": cfg, "roofline": roofline, "call_roofline": call_roofline,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "kernels": kernels,
                "clocks": clocks,
                "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                            "p10": sorted(step_ms)[len(step_ms) // 10],
                            "p90": sorted(step_ms)[(9 * len(step_ms)) // 10]}}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.which == "bwd":
        run_bwd(args)
    elif args.workload.startswith("decode"):
        run_decode(args)
    else:
        run_gdr(args)


if __name__ == "__main__":
    main()
