"""The seeded input recipe of every workload (the shapes and distributions of
the workloads the method is measured on): q and k L2-normalised per token
and head before the cast, beta in (0, 1), g a log-sigmoid (so g <= 0 and the
per-token decay exp(g) is in (0, 1)), varlen lengths within their bounds,
the same draw for the same seed."""
import pytest
import torch

from chunked_gated_delta_rule_gb300 import synthetic

W = synthetic.WORKLOADS


@pytest.mark.parametrize("name", sorted(W))
def test_workload_recipe(name):
    w = W[name]
    if w.T > 8192:  # the long workloads at a shorter length, same recipe
        w = synthetic.small(w, T=4096)
    x = synthetic.make_inputs(w)
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    assert x["q"].shape == (B, T, H, K) and x["k"].shape == (B, T, H, K)
    assert x["v"].shape == (B, T, H, V) and x["g"].shape == (B, T, H)
    assert x["q"].dtype == synthetic.torch_dtype(w.dtype) and x["g"].dtype == torch.float32
    tol = 1e-5 if w.dtype == "f32" else 1e-2  # the norm after the cast to 16 bits
    for t in (x["q"], x["k"]):
        n = t.float().norm(dim=-1)
        assert torch.allclose(n, torch.ones_like(n), atol=tol)
    assert (x["g"] <= 0).all() and torch.isfinite(x["g"]).all()
    if w.delta:
        assert x["beta"].shape == (B, T, H)
        assert ((x["beta"] > 0) & (x["beta"] < 1)).all()
    else:
        assert x["beta"] is None
    if w.n_seqs:
        cu = x["cu_seqlens"]
        lens = cu[1:] - cu[:-1]
        assert cu[0] == 0 and cu[-1] == T and N == w.n_seqs and B == 1
        rest = torch.ones_like(lens, dtype=torch.bool)
        if w.long_len:  # the skewed batch: its middle sequence has long_len tokens
            assert lens[w.n_seqs // 2] == w.long_len
            rest[w.n_seqs // 2] = False
        assert ((lens[rest] >= w.len_lo) & (lens[rest] <= w.len_hi)).all()
    else:
        assert x["cu_seqlens"] is None and N == B
    assert (x["h0"] is not None) == w.with_h0
    if w.with_h0:
        assert x["h0"].shape == (N, H, K, V)
    again = synthetic.make_inputs(w)
    for key in ("q", "k", "v", "g"):
        assert torch.equal(x[key], again[key]), key


def test_near_non_contracting_decay_of_the_64k_stress():
    """g = log sigmoid(N(6, 0.5)): a decay exp(g) of about 0.9975, the
    near non-contracting regime of the 64K context-parallel workload."""
    x = synthetic.make_inputs(synthetic.small(W["stress_64k_h8_bf16"], T=4096))
    decay = torch.exp(x["g"]).mean().item()
    assert 0.995 < decay < 0.999
