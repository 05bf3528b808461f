"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle

TOL_F32 = 1e-5   # relative L2, FP32 inputs
TOL_BF16 = 6e-3  # relative L2, BF16 inputs (o and ht)


def tol_of(x):
    return TOL_F32 if x["dtype"] == "f32" else TOL_BF16


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def run_gpu(x, **kw):
    import chunked_gated_delta_rule_gb300 as pkg
    d = to_dev(x)
    o, ht = pkg.gdr_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                              cu_seqlens=d["cu_seqlens"], h0=d["h0"], **kw)
    torch.cuda.synchronize()
    return o, ht


def run_oracle(x, pair_mask=None):
    o, ht, _ = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"],
                              cu_seqlens=x["cu_seqlens"], h0=x["h0"], pair_mask=pair_mask)
    return o, ht


def rel_l2_masked(x, ref):
    """Relative L2 over the entries the oracle computed (non-NaN)."""
    x = x.detach().cpu().to(torch.float64).numpy() if torch.is_tensor(x) else np.asarray(x)
    m = ~np.isnan(ref)
    d = np.linalg.norm((x[m] - ref[m]).ravel())
    r = np.linalg.norm(ref[m].ravel())
    return d / r if r > 0 else d


def sample_mask(N, H, pairs):
    m = np.zeros(N * H, dtype=bool)
    for n, h in pairs:
        m[n * H + h] = True
    return m
