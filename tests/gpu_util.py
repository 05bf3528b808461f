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


def max_seqlen(x):
    """The longest sequence's token count (the planning hint a caller that
    holds cu_seqlens on the host passes), None when dense."""
    cu = x["cu_seqlens"]
    if cu is None:
        return None
    return int((cu[1:] - cu[:-1]).max()) if cu.numel() > 1 else 0


def run_gpu(x, **kw):
    import chunked_gated_delta_rule_gb300 as pkg
    d = to_dev(x)
    kw.setdefault("max_seqlen", max_seqlen(x))
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


def seq_rows(x):
    """(first, end) rows of each sequence along the flattened B*T token axis."""
    if x["cu_seqlens"] is not None:
        cu = [int(c) for c in x["cu_seqlens"].tolist()]
        return list(zip(cu[:-1], cu[1:]))
    return [(n * x["T"], (n + 1) * x["T"]) for n in range(x["B"])]


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy() if torch.is_tensor(t) else np.asarray(t)


def worst_pair_rel_l2(x, o, ht, ro, rht):
    """The largest relative L2 over (sequence, head) pairs, for o (the pair's
    tokens) and for ht (the pair's state), over the pairs the oracle computed
    (NaN entries of a sampled reference are skipped).  A fault confined to a
    few tokens or one head, small in the whole-tensor norm, shows here."""
    H = x["H"]
    o64, ro64 = _f64(o), np.asarray(ro)
    o64 = o64.reshape(-1, H, o64.shape[-1])
    ro64 = ro64.reshape(-1, H, ro64.shape[-1])
    worst_o = worst_h = 0.0
    for n, (a, b) in enumerate(seq_rows(x)):
        for h in range(H):
            if b > a:
                r = ro64[a:b, h]
                if not np.isnan(r).all():
                    worst_o = max(worst_o, rel_l2_masked(o64[a:b, h], r))
            if ht is not None and rht is not None:
                r = np.asarray(rht)[n, h]
                if not np.isnan(r).all():
                    worst_h = max(worst_h, rel_l2_masked(_f64(ht[n, h]), r))
    return worst_o, worst_h


def assert_parity(x, o, ht, ro, rht, tol_o, tol_h=None, label=""):
    """Relative L2 against the oracle within the bar, over the whole tensors
    and for every (sequence, head) pair on its own.  Returns (whole o, whole
    ht, worst-pair o, worst-pair ht)."""
    tol_h = tol_o if tol_h is None else tol_h
    eo = rel_l2_masked(o, ro)
    eh = rel_l2_masked(ht, rht) if ht is not None else 0.0
    wo, wh = worst_pair_rel_l2(x, o, ht, ro, rht)
    print(f"{label}: rel_l2 o={eo:.3e} ht={eh:.3e}; worst pair o={wo:.3e} ht={wh:.3e}")
    assert eo <= tol_o and eh <= tol_h, (label, eo, eh)
    assert wo <= tol_o and wh <= tol_h, (label, "worst (sequence, head) pair", wo, wh)
    return eo, eh, wo, wh
