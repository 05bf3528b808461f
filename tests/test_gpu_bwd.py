"""GPU parity of the backward pass (gdr_chunk_bwd, through the C ABI)
against the FP64 oracle's gradients of L = <do, o> + <dht, ht>.

Tolerances (rel-L2 per gradient): FP32 inputs 1e-5 for every gradient, the
forward pass's FP32 bar.  BF16 inputs: dq, dk, dv are returned in BF16, one
rounding of an FP32 result (at most 2^-9 relative per element, about 1.7e-3
in rel-L2 measured), so they take the forward's BF16 bar 6e-3; dg, dbeta,
dh0 are FP32 arithmetic on the exact BF16 values the oracle also reads, so
they keep 1e-5.  FP16 inputs: dq, dk, dv rounded to FP16 once (2^-11), 2e-3;
the rest 1e-5.  The oracle reads the inputs after rounding to the input
dtype, so the comparison measures the kernels' arithmetic only.

The tensor-core route (BF16, K = V = 128, delta rule, serial or split into
segments; force_path=2, and the plan's choice for those shapes) computes
with BF16 operands in its forward recompute and reverse scan, and with
FP32 operands carried as BF16 hi + lo pairs in its per-chunk products:
every gradient is held to 1e-2, two sets of BF16 operand roundings of the
kind the forward's 6e-3 bar covers once.  The other tests here pin the CUDA-core route
(force_path=1), whose bars are the FP32 ones above.
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_rule_gb300 import synthetic

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
RAGGED = [1, 63, 64, 65, 127, 128, 257, 7, 300, 0]


TOL_TC = 1e-2  # every gradient of the tensor-core route


def tols(x, route=1):
    if route == 2:
        return {name: TOL_TC for name in NAMES}
    rounded = {"f32": 1e-5, "bf16": 6e-3, "f16": 2e-3}[x["dtype"]]
    return {"dq": rounded, "dk": rounded, "dv": rounded, "dg": 1e-5, "dbeta": 1e-5, "dh0": 1e-5}


def grads_in(x, seed=7, with_dht=True):
    """The incoming gradients: do in the input dtype, dht FP32 (seeded)."""
    gen = torch.Generator().manual_seed(seed)
    n = x["N"] if x["cu_seqlens"] is not None else x["B"]
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype)
    dht = torch.randn(n, x["H"], x["K"], x["V"], generator=gen) if with_dht else None
    return do, dht


def run_bwd(x, do, dht, layout="kv", **kw):
    """The backward on the GPU; the CUDA-core route unless force_path says
    otherwise."""
    import chunked_gated_delta_rule_gb300 as pkg
    kw.setdefault("force_path", 1)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    h0, dhtd = d["h0"], None if dht is None else dht.cuda()
    if layout == "vk":
        h0 = None if h0 is None else h0.transpose(-1, -2).contiguous()
        dhtd = None if dhtd is None else dhtd.transpose(-1, -2).contiguous()
    out = pkg.gdr_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do.cuda(),
                            cu_seqlens=d["cu_seqlens"], h0=h0, dht=dhtd, state_layout=layout,
                            **kw)
    torch.cuda.synchronize()
    out = list(out)
    if layout == "vk" and out[5] is not None:
        out[5] = out[5].transpose(-1, -2)
    return out


def check(x, with_dht=True, layout="kv", pair_mask=None, **kw):
    do, dht = grads_in(x, with_dht=with_dht)
    out = run_bwd(x, do, dht, layout=layout, **kw)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=x["cu_seqlens"],
                          h0=x["h0"], do=do, dht=dht, pair_mask=pair_mask)
    tol = tols(x, kw.get("force_path", 1))
    errs = {}
    for name, a, r in zip(NAMES, out, ref):
        if r is None:
            assert a is None, name
            continue
        a = a.detach().cpu().to(torch.float64).numpy()
        m = ~np.isnan(r)
        assert np.isfinite(a).all(), name
        num = np.linalg.norm((a[m] - r[m]).ravel())
        den = np.linalg.norm(r[m].ravel())
        errs[name] = num / den if den > 0 else num
    bad = {k: v for k, v in errs.items() if not v <= tol[k]}
    assert not bad, (bad, errs)
    return errs


def test_tiny_dense_f32():
    """FP32, B=1, T=256, H=2, K=V=64, h0 and dht."""
    check(synthetic.make_inputs(W["tiny_dense_f32"]))


@pytest.mark.parametrize("K,V", [(16, 16), (32, 48), (128, 64), (256, 128), (64, 256)])
def test_f32_shapes(K, V):
    w = synthetic.small(W["tiny_dense_f32"], K=K, V=V, T=150, H=2, B=2)
    check(synthetic.make_inputs(w))


def test_bf16_varlen_ragged_and_empty():
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    check(synthetic.make_inputs(w, lengths=RAGGED))


def test_bf16_without_dht_or_h0():
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    check(synthetic.make_inputs(w, lengths=[65, 130, 7]), with_dht=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_beta_free(dtype):
    w = synthetic.small(W["gla_k256_v512_bf16"], B=1, T=300, H=2, V=256, dtype=dtype)
    check(synthetic.make_inputs(w))


def test_state_layout_vk_and_h0():
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    check(synthetic.make_inputs(w, lengths=[70, 5, 129]), layout="vk")


def test_f16_inputs():
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True, dtype="f16")
    check(synthetic.make_inputs(w, lengths=[70, 5, 129]))


def test_int64_seqlens_match_int32():
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[70, 5, 0, 129])
    do, dht = grads_in(x)
    a = run_bwd(x, do, dht)
    x64 = dict(x, cu_seqlens=x["cu_seqlens"].to(torch.int64))
    b = run_bwd(x64, do, dht)
    for name, u, v in zip(NAMES, a, b):
        assert torch.equal(u, v), name


def test_bit_identical_repeats_and_poisoned_outputs_written():
    """Two calls give the same bits, and every element of NaN-filled output
    buffers is written (including the tokens of one-token sequences)."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[1, 64, 65, 200])
    do, dht = grads_in(x)
    nan = lambda t, dt=None: torch.full(t.shape, float("nan"), dtype=dt or t.dtype, device="cuda")
    bufs = dict(dq=nan(x["q"]), dk=nan(x["k"]), dv=nan(x["v"]), dg=nan(x["g"]),
                dbeta=nan(x["beta"]), dh0=nan(x["h0"]))
    a = run_bwd(x, do, dht, **bufs)
    for name, t in zip(NAMES, a):
        assert torch.isfinite(t.float()).all(), name
    b = run_bwd(x, do, dht)
    for name, u, v in zip(NAMES, a, b):
        assert torch.equal(u, v), name


def test_caller_workspace_matches_internal_allocation():
    import chunked_gated_delta_rule_gb300 as pkg
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=[65, 130, 7])
    do, dht = grads_in(x)
    nbytes = pkg.gdr_bwd_workspace_size(1, x["T"], 2, 128, 128, N=3)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    a = run_bwd(x, do, dht)
    b = run_bwd(x, do, dht, workspace=ws)
    for name, u, v in zip(NAMES, a, b):
        assert torch.equal(u, v), name
    with pytest.raises(pkg.GdrError):
        run_bwd(x, do, dht, workspace=ws[: nbytes // 2])


@pytest.mark.parametrize("name", ["wide_varlen_bf16", "long_16k_bf16", "gla_k256_v512_bf16"])
def test_full_size_sampled_pairs(name):
    """Full-size workloads; the oracle computes three (sequence, head) pairs
    (first, middle, last), the other pairs are checked to be finite."""
    x = synthetic.make_inputs(W[name])
    n = x["N"] if x["cu_seqlens"] is not None else x["B"]
    pairs = n * x["H"]
    mask = np.zeros(pairs, dtype=bool)
    mask[[0, pairs // 2, pairs - 1]] = True
    check(x, pair_mask=mask)


@pytest.mark.parametrize("S", [2, 4, 16, 64])
@pytest.mark.parametrize("case", ["bf16_varlen_h0", "f32_k64", "f32_k256", "beta_free"])
def test_segment_split(case, S):
    """The forward recompute and the reverse scan split into S segments: the
    pre-scan, the ordered composition from the last segment to the first (the
    delta-rule composition at K <= 128, the generic one at K = 256, the
    scalar one for beta-free) and the output pass give the same gradients
    within the tolerances."""
    if case == "bf16_varlen_h0":
        w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
        x = synthetic.make_inputs(w, lengths=[700, 65, 1, 300, 0])
    elif case == "f32_k64":
        x = synthetic.make_inputs(synthetic.small(W["tiny_dense_f32"], T=900, B=2))
    elif case == "f32_k256":
        x = synthetic.make_inputs(synthetic.small(W["tiny_dense_f32"], K=256, V=64, T=600))
    else:
        x = synthetic.make_inputs(synthetic.small(W["gla_k256_v512_bf16"], B=1, T=1000, H=2,
                                                  V=128))
    check(x, n_segments=S)


def test_long_single_sequence_split_matches_oracle():
    """One 4096-token sequence, one head (the low-wave shape the split is
    for), automatic plan, against the oracle."""
    w = synthetic.small(W["stress_64k_h1_bf16"], T=4096)
    check(synthetic.make_inputs(w))


@pytest.mark.parametrize("combo", ["vk_layout", "int64_seqlens", "f16"])
def test_split_with_layout_and_dtype_options(combo):
    """The segment split combined with the transposed state layout (dht in,
    dh0 out through the reverse composition), int64 cu_seqlens and FP16
    inputs."""
    dtype = "f16" if combo == "f16" else "bf16"
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True, dtype=dtype)
    x = synthetic.make_inputs(w, lengths=[700, 65, 1, 300])
    if combo == "int64_seqlens":
        x = dict(x, cu_seqlens=x["cu_seqlens"].to(torch.int64))
    check(x, layout="vk" if combo == "vk_layout" else "kv", n_segments=4)


# --------------------------------------------------------------------------
# the tensor-core route
# --------------------------------------------------------------------------
def _bits(t):
    return None if t is None else t.detach().contiguous().view(torch.uint8).cpu()


def test_tc_route_varlen_ragged_empty_h0_dht():
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    print(check(synthetic.make_inputs(w, lengths=RAGGED), force_path=2))


def test_tc_route_without_dht_or_h0():
    w = synthetic.small(W["wide_varlen_bf16"], H=3)
    print(check(synthetic.make_inputs(w, lengths=[200, 64, 1, 129]), with_dht=False,
                force_path=2))


def test_tc_route_state_layout_vk_dense_batch():
    w = synthetic.small(W["long_16k_bf16"], B=2, T=700, H=2, with_h0=True)
    print(check(synthetic.make_inputs(w), layout="vk", force_path=2))


@pytest.mark.parametrize("name", ["wide_varlen_bf16", "long_16k_bf16"])
def test_tc_route_full_size_sampled_pairs(name):
    x = synthetic.make_inputs(W[name])
    n = x["N"] if x["cu_seqlens"] is not None else x["B"]
    pairs = n * x["H"]
    mask = np.zeros(pairs, dtype=bool)
    mask[[0, pairs // 2, pairs - 1]] = True
    print(check(x, pair_mask=mask, force_path=2))


def test_tc_route_is_the_default_for_its_shapes_and_bits_do_not_depend_on_the_grid():
    """BF16, K = V = 128, delta rule, serial: the plan takes the tensor-core
    route; its gradients are the same bits at any grid of the persistent
    kernels and from run to run."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[300, 65, 7, 129])
    do, dht = grads_in(x)
    ref = run_bwd(x, do, dht, force_path=2)
    for kw in (dict(force_path=0), dict(force_path=2, grid_limit=1),
               dict(force_path=2, grid_limit=7), dict(force_path=2)):
        out = run_bwd(x, do, dht, **kw)
        for name, a, b in zip(NAMES, out, ref):
            assert (a is None) == (b is None), name
            if a is not None:
                assert torch.equal(_bits(a), _bits(b)), (name, kw)


# the tensor-core route split into segments: the forward's pre-scan,
# composition and an output pass keeping the images, then the reverse
# scan's offsets from E = 0, the composition from dht to dh0 over the
# transposed forward maps and its output pass
@pytest.mark.parametrize("S", [2, 5])
def test_tc_route_segments_varlen_ragged(S):
    """Sequences with fewer chunks than segments (their empty segments are
    skipped and the reversed summary slots count the others), h0 and dht."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[700, 65, 1, 300, 129])
    print(check(x, force_path=2, n_segments=S))


def test_tc_route_segments_state_layout_vk_without_dht():
    w = synthetic.small(W["long_16k_bf16"], B=2, T=1000, H=2, with_h0=True)
    print(check(synthetic.make_inputs(w), layout="vk", with_dht=False, force_path=2,
                n_segments=4))


def test_tc_route_segments_bits_do_not_depend_on_the_grid():
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[900, 65, 7, 300])
    do, dht = grads_in(x)
    ref = run_bwd(x, do, dht, force_path=2, n_segments=4)
    for kw in (dict(grid_limit=1), dict(grid_limit=7), dict()):
        out = run_bwd(x, do, dht, force_path=2, n_segments=4, **kw)
        for name, a, b in zip(NAMES, out, ref):
            if a is not None:
                assert torch.equal(_bits(a), _bits(b)), (name, kw)


@pytest.mark.parametrize("name,pairs", [("stress_64k_h8_bf16", (0, 7)),
                                        ("stress_64k_h1_bf16", (0,))])
def test_tc_route_plan_split_full_size_sampled_pairs(name, pairs):
    """64K tokens at the plan's segment count (the route's default)."""
    x = synthetic.make_inputs(W[name])
    mask = np.zeros(x["B"] * x["H"], dtype=bool)
    mask[list(pairs)] = True
    print(check(x, pair_mask=mask, force_path=2))
