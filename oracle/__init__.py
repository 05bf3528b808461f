"""CPU FP64 oracle for the chunked gated-delta-rule forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` import this package.  The CUDA
library never imports, links or calls it, and it imports nothing from the
CUDA library.

The arithmetic lives in ``gdr_oracle.c`` (plain C, FP64, token by token):

* :func:`forward` -- the per-token recurrence
  ``S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T``,
  ``o_t = S_t q_t / sqrt(K)`` (state recurrence of cuLA PR #127 "Summary";
  the scan of fla's ``chunk_gated_delta_rule_fwd_kernel_h_blockdim64``, Kev
  PR #259 intro), with ``beta=None`` selecting the beta-free gated linear
  attention write ``S_t = alpha_t S_{t-1} + v_t k_t^T``.
* :func:`backward` -- the gradient of :func:`forward` for the loss
  ``<do, o> + <dht, ht>`` with respect to q, k, v, g, beta and h0: reverse-mode
  differentiation of each token step, the state gradient dH running backward
  through the sequence (the reverse dH recurrence of the flash-linear-attention
  ABC issue #23 pages, "Problem" and "Proposed Dataflow" step 4; gradients
  dQ/dK/dV and of the states, its "Fixture-First Correctness Contract").
* :func:`affine` -- the affine map ``h_out = M h_in + c`` of that recurrence
  over a token range (the per-segment summary of cuLA PR #127 "Root cause and
  implementation").
* :func:`forward_segmented` -- the serial result rebuilt from per-segment
  summaries composed in order (same page), used to pin the segment split.

Pins for every function: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgdr_oracle.so")

_lib = None
_lock = threading.Lock()

CHUNK = 64


def build(force: bool = False) -> str:
    """Compile ``gdr_oracle.c`` with gcc into ``oracle/_build``.  Plain -O2, no
    fast-math, no machine-specific flags (the same source builds on x86-64
    and aarch64)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled copy of ``gdr_oracle.c`` and declare its entry points.
    The tests use this to open deliberately broken copies (mutants) and show
    that the pins reject them."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.gdr_oracle_fwd.restype = ctypes.c_int
    lib.gdr_oracle_fwd.argtypes = [
        dp, dp, dp, dp, dp, i64p, dp, dp, dp,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        ctypes.POINTER(ctypes.c_uint8), ctypes.c_int]
    lib.gdr_oracle_bwd.restype = ctypes.c_int
    lib.gdr_oracle_bwd.argtypes = [
        dp, dp, dp, dp, dp, i64p, dp, dp, dp, dp, dp, dp, dp, dp, dp,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        ctypes.POINTER(ctypes.c_uint8), ctypes.c_int]
    lib.gdr_oracle_affine.restype = ctypes.c_int
    lib.gdr_oracle_affine.argtypes = [
        dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, dp, dp]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f64(x):
    """Any array-like (numpy, torch CPU/GPU tensor of any float dtype) to a
    C-contiguous float64 numpy array.  BF16 values upcast exactly."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def forward(q, k, v, g, beta=None, cu_seqlens=None, h0=None, scale=None,
            want_ht=True, pair_mask=None, n_threads=0, lib=None):
    """Token-by-token FP64 forward pass.

    Shapes: q, k [B,T,H,K]; v [B,T,H,V]; g, beta [B,T,H]; h0 [N,H,K,V];
    cu_seqlens [N+1] (varlen, B == 1).  Returns ``(o, ht, threads_used)`` with
    o [B,T,H,V] and ht [N,H,K,V] (None if ``want_ht`` is false), FP64.
    ``pair_mask`` ([N*H] bool) limits the work to some (sequence, head) pairs;
    the other pairs' outputs are NaN.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta, h0 = _f64(beta), _f64(h0)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        N = cu.shape[0] - 1
    else:
        cu = None
        N = B
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    o = np.full((B, T, H, V), np.nan)
    ht = np.full((N, H, K, V), np.nan) if want_ht else None
    mask = None
    if pair_mask is not None:
        mask = np.ascontiguousarray(np.asarray(pair_mask, dtype=np.uint8).reshape(-1))
        assert mask.shape[0] == N * H
    lib = lib or _load()
    r = lib.gdr_oracle_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(cu, ctypes.c_int64), _ptr(h0), _ptr(o), _ptr(ht),
        B, T, H, K, V, N, float(scale), _ptr(mask, ctypes.c_uint8),
        int(n_threads))
    if r < 0:
        raise ValueError("gdr_oracle_fwd rejected its arguments")
    return o, ht, r


def backward(q, k, v, g, beta=None, cu_seqlens=None, h0=None, do=None, dht=None,
             scale=None, pair_mask=None, n_threads=0, lib=None):
    """Token-by-token FP64 gradients of ``L = <do, o> + <dht, ht>``.

    Shapes as for :func:`forward`; ``do`` [B,T,H,V], ``dht`` [N,H,K,V] or
    None (no final-state term).  Returns ``(dq, dk, dv, dg, dbeta, dh0)``,
    FP64, ``dbeta`` None in the beta-free mode.  ``pair_mask`` limits the work
    to some (sequence, head) pairs; the other pairs' gradients are NaN.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta, h0, do, dht = _f64(beta), _f64(h0), _f64(do), _f64(dht)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        N = cu.shape[0] - 1
    else:
        cu = None
        N = B
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    dq = np.full((B, T, H, K), np.nan)
    dk = np.full((B, T, H, K), np.nan)
    dv = np.full((B, T, H, V), np.nan)
    dg = np.full((B, T, H), np.nan)
    dbeta = np.full((B, T, H), np.nan) if beta is not None else None
    dh0 = np.full((N, H, K, V), np.nan)
    mask = None
    if pair_mask is not None:
        mask = np.ascontiguousarray(np.asarray(pair_mask, dtype=np.uint8).reshape(-1))
        assert mask.shape[0] == N * H
    r = (lib or _load()).gdr_oracle_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu, ctypes.c_int64),
        _ptr(h0), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
        _ptr(dbeta), _ptr(dh0), B, T, H, K, V, N, float(scale),
        _ptr(mask, ctypes.c_uint8), int(n_threads))
    if r < 0:
        raise ValueError("gdr_oracle_bwd rejected its arguments")
    return dq, dk, dv, dg, dbeta, dh0


def affine(k, v, g, beta=None, lib=None):
    """Affine map of the recurrence over one token range of one (sequence,
    head): ``h_out = M @ h_in + c``.  k [L,K], v [L,V], g [L], beta [L] or
    None.  Returns (M [K,K], c [K,V]) in FP64."""
    k, v, g, beta = _f64(k), _f64(v), _f64(g), _f64(beta)
    L, K = k.shape
    V = v.shape[1]
    M = np.empty((K, K))
    c = np.empty((K, V))
    r = (lib or _load()).gdr_oracle_affine(_ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  L, K, V, K, V, 1, _ptr(M), _ptr(c))
    if r != 0:
        raise ValueError("gdr_oracle_affine rejected its arguments")
    return M, c


def segment_bounds(n_tokens: int, n_segments: int, chunk: int = CHUNK, per=None):
    """Token ranges of the segments of one sequence: runs of
    ceil(n_chunks / S) whole 64-token chunks; a sequence with fewer chunks
    than S uses fewer segments (the reading taken where the pages leave the
    split rule open).  ``per`` fixes the run length in chunks instead (one
    common length for a whole batch, the other reading of that rule)."""
    n_chunks = -(-n_tokens // chunk)
    if n_chunks == 0:
        return []
    if per is None:
        per = -(-n_chunks // max(1, n_segments))
    out = []
    c0 = 0
    while c0 < n_chunks:
        c1 = min(n_chunks, c0 + per)
        out.append((c0 * chunk, min(n_tokens, c1 * chunk)))
        c0 = c1
    return out


def forward_segmented(q, k, v, g, beta=None, cu_seqlens=None, h0=None,
                      n_segments=2, scale=None, lib=None, common=False):
    """Serial result rebuilt through the segment split: per (sequence, head)
    each segment's affine summary (M_s, c_s) from :func:`affine`, the ordered
    composition h_{s+1} = M_s h_s + c_s, then each segment's outputs from its
    composed initial state by :func:`forward`.  ``common``: every sequence
    cut into runs of ceil(longest sequence's chunks / S) chunks, a shorter
    sequence left as one run.  Returns (o, ht)."""
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    beta, h0 = _f64(beta), _f64(h0)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = [int(x) for x in np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens)]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    else:
        spans = [(b, 0, T) for b in range(B)]
    N = len(spans)
    o = np.full((B, T, H, V), np.nan)
    ht = np.zeros((N, H, K, V))
    per = None
    if common:
        longest = max([-(-(t1 - t0) // CHUNK) for (_, t0, t1) in spans] + [0])
        per = max(1, -(-longest // max(1, n_segments)))
    for n, (row, t0, t1) in enumerate(spans):
        for hh in range(H):
            h = h0[n, hh].copy() if h0 is not None else np.zeros((K, V))
            for (s0, s1) in segment_bounds(t1 - t0, n_segments, per=per):
                a, b = t0 + s0, t0 + s1
                sl = (slice(row, row + 1), slice(a, b), slice(hh, hh + 1))
                bo, _, _ = forward(q[sl], k[sl], v[sl], g[sl],
                                   None if beta is None else beta[sl],
                                   h0=h[None, None], scale=scale,
                                   want_ht=False, n_threads=1, lib=lib)
                o[row, a:b, hh] = bo[0, :, 0]
                M, c = affine(k[row, a:b, hh], v[row, a:b, hh], g[row, a:b, hh],
                              None if beta is None else beta[row, a:b, hh],
                              lib=lib)
                h = M @ h + c
            ht[n, hh] = h
    return o, ht


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, in FP64."""
    x, ref = _f64(x), _f64(ref)
    num = float(np.linalg.norm((x - ref).reshape(-1)))
    den = float(np.linalg.norm(ref.reshape(-1)))
    return num / den if den > 0 else num
