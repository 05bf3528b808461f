"""The differentiable entry point (chunk_gated_delta_rule): torch autograd
through the library's forward and backward passes, checked against the FP64
oracle's gradients of the same loss (tolerances of test_gpu_bwd.py: BF16
delta-rule inputs at K = V = 128 take the tensor-core route, 1e-2 for every
gradient)."""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_rule_gb300 import synthetic

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS


def _rel(a, r):
    a = a.detach().cpu().to(torch.float64).numpy()
    return np.linalg.norm((a - r).ravel()) / np.linalg.norm(r.ravel())


@pytest.mark.parametrize("case", ["bf16_varlen_h0", "f32_dense_no_state", "bf16_beta_free"])
def test_autograd_matches_oracle(case):
    import chunked_gated_delta_rule_gb300 as pkg
    if case == "bf16_varlen_h0":
        x = synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True),
                                  lengths=[70, 5, 129])
        want_state, tol = True, (1e-2, 1e-2)
    elif case == "f32_dense_no_state":
        x = synthetic.make_inputs(synthetic.small(W["tiny_dense_f32"], with_h0=False, B=2, T=150))
        want_state, tol = False, (1e-5, 1e-5)
    else:
        x = synthetic.make_inputs(synthetic.small(W["gla_k256_v512_bf16"], B=1, T=200, H=2,
                                                  V=128))
        want_state, tol = True, (6e-3, 1e-5)
    gen = torch.Generator().manual_seed(3)
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype)
    n = x["N"] if x["cu_seqlens"] is not None else x["B"]
    dht = torch.randn(n, x["H"], x["K"], x["V"], generator=gen) if want_state else None
    leaf = {}
    for name in ("q", "k", "v", "g", "beta", "h0"):
        t = x[name]
        leaf[name] = None if t is None else t.cuda().requires_grad_(True)
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cuda()
    o, ht = pkg.chunk_gated_delta_rule(leaf["q"], leaf["k"], leaf["v"], leaf["g"], leaf["beta"],
                                       initial_state=leaf["h0"], output_final_state=want_state,
                                       cu_seqlens=cu)
    assert (ht is not None) == want_state
    loss = (o.float() * do.cuda().float()).sum()
    if want_state:
        loss = loss + (ht * dht.cuda()).sum()
    loss.backward()
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=x["cu_seqlens"],
                          h0=x["h0"], do=do, dht=dht)
    for i, name in enumerate(("q", "k", "v", "g", "beta", "h0")):
        if leaf[name] is None:
            continue
        bound = tol[0] if name in ("q", "k", "v") else tol[1]
        err = _rel(leaf[name].grad, ref[i])
        assert err <= bound, (name, err)
