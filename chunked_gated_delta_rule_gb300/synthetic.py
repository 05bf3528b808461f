"""Seeded synthetic inputs for the chunked gated-delta-rule forward pass.

This module only draws random tensors.  It holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may take their inputs
from it.

Recipe (one CPU ``torch.Generator`` per draw, seeded; draw order: lengths
(varlen only), q, k, v, beta logits (delta mode only), gate logits, h0):

* q, k ~ N(0, 1), then L2-normalised over the key dim per token and head, in
  FP32 before any cast;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1));
* g = log(sigmoid(N(mu, sigma))) per token and head (mu = 3, sigma = 1; the
  near non-contracting stress workload uses mu = 6, sigma = 0.5);
* h0 ~ 0.1 * N(0, 1) where an initial state is passed;
* a skewed batch draws its lengths like the others, then sets the middle
  sequence's length to ``long_len``;
* q, k, v are then cast to the workload dtype (BF16 or FP32); g, beta, h0
  stay FP32.

Workloads (sizes as the project statement fixes them; the pages measure on
no public dataset -- the fla/Kev question rows and the cuLA 64K reproducer
are stood in for by these):
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch
import torch.nn.functional as F


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int                 # tokens per batch row (ignored when varlen)
    H: int
    K: int
    V: int
    dtype: str             # "f32" | "bf16" | "f16" (q, k, v, o)
    n_seqs: int = 0        # > 0: varlen, lengths U{len_lo..len_hi}, packed
    len_lo: int = 0
    len_hi: int = 0
    g_mu: float = 3.0
    g_sigma: float = 1.0
    delta: bool = True     # False: beta-free (beta=None)
    with_h0: bool = False
    seed: int = 0
    long_len: int = 0      # > 0: sequence n_seqs // 2 has this length instead


WORKLOADS = {
    # FP32 tiny dense case, small enough for brute-force checks.
    "tiny_dense_f32": Workload("tiny_dense_f32", 1, 256, 2, 64, 64, "f32",
                               with_h0=True),
    # Wide varlen batch: 32 packed sequences of 128..512 tokens.
    "wide_varlen_bf16": Workload("wide_varlen_bf16", 1, 0, 16, 128, 128,
                                 "bf16", n_seqs=32, len_lo=128, len_hi=512),
    # Long single state: one 16K-token sequence, 16 heads.
    "long_16k_bf16": Workload("long_16k_bf16", 1, 16384, 16, 128, 128, "bf16"),
    # 64K context-parallel stress, near non-contracting decay.
    "stress_64k_h8_bf16": Workload("stress_64k_h8_bf16", 1, 65536, 8, 128,
                                   128, "bf16", g_mu=6.0, g_sigma=0.5),
    "stress_64k_h1_bf16": Workload("stress_64k_h1_bf16", 1, 65536, 1, 128,
                                   128, "bf16", g_mu=6.0, g_sigma=0.5),
    # Beta-free (pure gated linear attention) geometry, K=256, V=512.
    "gla_k256_v512_bf16": Workload("gla_k256_v512_bf16", 2, 8192, 4, 256, 512,
                                   "bf16", delta=False, with_h0=True),
    # One 16K-token sequence among 100 of 128..512 tokens (the longest
    # sequence, not the mean, sets the serial scan's time).
    "skewed_varlen_bf16": Workload("skewed_varlen_bf16", 1, 0, 16, 128, 128, "bf16",
                                   n_seqs=101, len_lo=128, len_hi=512, long_len=16384),
    # The same skew with 4 heads and 31 short sequences: few chains besides
    # the long sequence's, so splitting it pays.
    "skewed_varlen_h4_bf16": Workload("skewed_varlen_h4_bf16", 1, 0, 4, 128, 128, "bf16",
                                      n_seqs=32, len_lo=128, len_hi=512, long_len=16384),
    # The same skew in the beta-free geometry (K = 256, V = 512, h0 in).
    "skewed_gla_h4_bf16": Workload("skewed_gla_h4_bf16", 1, 0, 4, 256, 512, "bf16",
                                   n_seqs=32, len_lo=128, len_hi=512, long_len=16384,
                                   delta=False, with_h0=True),
    # The wide varlen batch with FP16 q / k / v.
    "wide_varlen_f16": Workload("wide_varlen_f16", 1, 0, 16, 128, 128,
                                "f16", n_seqs=32, len_lo=128, len_hi=512),
    # Decode step: 256 sequences of one token each, every one continuing a
    # state held in a pool (gdr_recurrent_fwd).
    "decode_bf16": Workload("decode_bf16", 1, 0, 16, 128, 128, "bf16", n_seqs=256,
                            len_lo=1, len_hi=1, with_h0=True),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[name]


def make_inputs(w: Workload, lengths: Optional[list] = None, T: Optional[int] = None,
                beta_zero: bool = False) -> dict:
    """Draw one workload's inputs on the CPU.

    ``lengths`` forces explicit varlen lengths (tests of ragged tails);
    ``T`` overrides the dense length (reduced-size parity cases);
    ``beta_zero`` replaces beta by an all-zero tensor (the literal beta = 0
    check).  Returns a dict with q, k, v, g, beta (or None), cu_seqlens (int32
    or None), h0 (or None), and the shape numbers B, T, H, K, V, N.
    """
    gen = torch.Generator().manual_seed(w.seed)
    H, K, V = w.H, w.K, w.V
    cu = None
    if lengths is not None or w.n_seqs > 0:
        if lengths is None:
            lens = torch.randint(w.len_lo, w.len_hi + 1, (w.n_seqs,), generator=gen)
            if w.long_len:
                lens[w.n_seqs // 2] = w.long_len
        else:
            lens = torch.tensor(lengths, dtype=torch.int64)
        cu = torch.zeros(lens.numel() + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
        B, TT, N = 1, int(lens.sum()), int(lens.numel())
    else:
        B, TT = w.B, (T if T is not None else w.T)
        N = B
    q = torch.randn(B, TT, H, K, generator=gen)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    k = torch.randn(B, TT, H, K, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    v = torch.randn(B, TT, H, V, generator=gen)
    beta = None
    if w.delta:
        beta = torch.sigmoid(torch.randn(B, TT, H, generator=gen))
        if beta_zero:
            beta = torch.zeros_like(beta)
    g = F.logsigmoid(torch.randn(B, TT, H, generator=gen) * w.g_sigma + w.g_mu)
    h0 = 0.1 * torch.randn(N, H, K, V, generator=gen) if w.with_h0 else None
    dt = torch_dtype(w.dtype)
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(),
                v=v.to(dt).contiguous(), g=g.contiguous(),
                beta=None if beta is None else beta.contiguous(),
                cu_seqlens=cu, h0=h0, B=B, T=TT, H=H, K=K, V=V, N=N,
                dtype=w.dtype)


def small(w: Workload, **overrides) -> Workload:
    """A copy of a workload with some fields replaced (reduced-size cases)."""
    return dataclasses.replace(w, **overrides)


def make_state_pool(x: dict, n_states: int, seed: int = 1):
    """A pool of ``n_states`` states [P, H, K, V] holding each sequence's h0
    at a distinct seeded row, the other rows random; returns ``(pool,
    indices)`` with int32 ``indices[n]`` = the row of sequence n."""
    gen = torch.Generator().manual_seed(seed)
    N, H, K, V = x["N"], x["H"], x["K"], x["V"]
    if n_states < N:
        raise ValueError("the pool needs a row per sequence")
    idx = torch.randperm(n_states, generator=gen)[:N].to(torch.int32)
    pool = 0.1 * torch.randn(n_states, H, K, V, generator=gen)
    if x["h0"] is not None:
        pool[idx.long()] = x["h0"]
    return pool, idx
