"""Strided q, k, v and o at the boundary: views of one fused projection
([B, T, 3, H, K]), head-major views ([B, H, T, K] transposed), an output that
is a slice of a wider tensor.  Each runs in place (no copy), matches the FP64
oracle, and gives exactly the bits of the same call on contiguous copies
(both read the same values in the same order; only the addressing differs).
Strides that break TMA's 16-byte rule move the call to the CUDA-core path,
which then matches its own contiguous run bit for bit.  All calls go through
the C ABI."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import TOL_BF16, TOL_F32, assert_parity, max_seqlen, run_oracle, to_dev

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS


def _bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu()


def fused_views(x, pad=0):
    """q, k, v as views of one [B, T, 3, H, K + pad] tensor (K == V): token
    stride 3 H (K + pad), head stride K + pad."""
    B, T, H, K = x["q"].shape
    big = torch.zeros(B, T, 3, H, K + pad, dtype=x["q"].dtype, device="cuda")
    for j, name in enumerate(("q", "k", "v")):
        big[:, :, j, :, :K] = x[name].cuda()
    return big[:, :, 0, :, :K], big[:, :, 1, :, :K], big[:, :, 2, :, :K]


def run(d, q, k, v, o=None, **kw):
    o_, ht = pkg.gdr_chunk_fwd(q, k, v, d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                               h0=d["h0"], o=o, **kw)
    torch.cuda.synchronize()
    return o_, ht


def check_views(x, q, k, v, o=None, tol=TOL_BF16, **kw):
    d = to_dev(x)
    kw.setdefault("max_seqlen", max_seqlen(x))
    assert not q.is_contiguous()
    o_s, ht_s = run(d, q, k, v, o, **kw)
    o_c, ht_c = run(d, d["q"], d["k"], d["v"], **kw)
    assert torch.equal(_bits(o_s), _bits(o_c))
    assert torch.equal(_bits(ht_s), _bits(ht_c))
    ro, rht = run_oracle(x)
    assert_parity(x, o_s, ht_s, ro, rht, tol, label=f"strided {kw}")


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("S", [1, 3])
def test_fused_projection_delta_varlen(path, S):
    w = synthetic.small(W["wide_varlen_bf16"], H=3, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[1, 63, 64, 65, 200, 0, 131])
    q, k, v = fused_views(x)
    check_views(x, q, k, v, n_segments=S, force_path=path)


@pytest.mark.parametrize("path", [1, 2])
def test_fused_projection_dense_batch_and_strided_output(path):
    w = synthetic.small(W["long_16k_bf16"], B=2, T=300, H=2)
    x = synthetic.make_inputs(w)
    q, k, v = fused_views(x)
    wide = torch.full((2, 300, 2, 2 * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = wide[..., 128:]  # token stride 2 H V, head stride 2 V
    check_views(x, q, k, v, o=o, n_segments=2, force_path=path)
    assert torch.isnan(wide[..., :128].float()).all()  # nothing written outside o


def test_head_major_views_beta_free():
    """q, k, v stored head-major ([1, H, T, D], transposed to [1, T, H, D]):
    token stride D, head stride T D; the beta-free tensor-core scan."""
    w = synthetic.small(W["gla_k256_v512_bf16"], B=1, T=400, H=2, K=128, V=256)
    x = synthetic.make_inputs(w)
    hm = {n: x[n].cuda().transpose(1, 2).contiguous().transpose(1, 2) for n in ("q", "k", "v")}
    check_views(x, hm["q"], hm["k"], hm["v"], n_segments=2)


def test_fp32_fused_projection():
    w = synthetic.small(W["tiny_dense_f32"], T=200)
    x = synthetic.make_inputs(w)
    q, k, v = fused_views(x)
    check_views(x, q, k, v, tol=TOL_F32)


def test_strides_off_the_tma_grid_take_the_cuda_core_path():
    """A padded row of 132 BF16 (264 bytes, not a multiple of 16): the plan
    moves the call to the CUDA-core path, bit-identical to that path's
    contiguous run and within the BF16 bar."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=[70, 129])
    q, k, v = fused_views(x, pad=4)
    d = to_dev(x)
    o_s, ht_s = run(d, q, k, v)
    o_c, ht_c = run(d, d["q"], d["k"], d["v"], force_path=1)
    assert torch.equal(_bits(o_s), _bits(o_c)) and torch.equal(_bits(ht_s), _bits(ht_c))
    ro, rht = run_oracle(x)
    assert_parity(x, o_s, ht_s, ro, rht, TOL_BF16, label="padded rows")


def test_recurrent_strided_inputs():
    w = synthetic.small(W["decode_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=[1, 3, 0, 2])
    pool, idx = synthetic.make_state_pool(x, 6)
    q, k, v = fused_views(x)
    d = to_dev(x)
    outs = []
    for args in ((q, k, v), (d["q"], d["k"], d["v"])):
        p = pool.cuda()
        o = pkg.gdr_recurrent_fwd(*args, d["g"], d["beta"], cu_seqlens=d["cu_seqlens"], state=p,
                                  state_indices=idx.cuda())
        torch.cuda.synchronize()
        outs.append((o, p))
    assert torch.equal(_bits(outs[0][0]), _bits(outs[1][0]))
    assert torch.equal(_bits(outs[0][1]), _bits(outs[1][1]))


def test_backward_reads_strided_inputs():
    """gdr_chunk_bwd on views of a fused projection: the gradients are the
    bits of the contiguous call."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[65, 130, 7])
    q, k, v = fused_views(x)
    d = to_dev(x)
    gen = torch.Generator().manual_seed(7)
    do = torch.randn(x["v"].shape, generator=gen).to(torch.bfloat16).cuda()
    dht = torch.randn(x["h0"].shape, generator=gen).cuda()
    res = []
    for args in ((q, k, v), (d["q"], d["k"], d["v"])):
        res.append(pkg.gdr_chunk_bwd(*args, d["g"], d["beta"], do, cu_seqlens=d["cu_seqlens"],
                                     h0=d["h0"], dht=dht))
        torch.cuda.synchronize()
    for a, b in zip(*res):
        assert torch.equal(_bits(a), _bits(b))


def test_autograd_on_fused_projection_views():
    """chunk_gated_delta_rule takes the views as they are; the gradient
    reaches the fused tensor through them."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=[100, 30])
    B, T, H, K = x["q"].shape
    big = torch.zeros(B, T, 3, H, K, dtype=torch.bfloat16, device="cuda")
    for j, n in enumerate(("q", "k", "v")):
        big[:, :, j] = x[n].cuda()
    big.requires_grad_(True)
    d = to_dev(x)
    o, _ = pkg.chunk_gated_delta_rule(big[:, :, 0], big[:, :, 1], big[:, :, 2], d["g"], d["beta"],
                                      cu_seqlens=d["cu_seqlens"])
    o.float().sum().backward()
    assert big.grad is not None and torch.isfinite(big.grad.float()).all()
    o_c, _ = pkg.gdr_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(_bits(o.detach()), _bits(o_c))
