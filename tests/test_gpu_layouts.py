"""The layout flags of gdr_dims (include/gdr.h gdr_flags): int64 cu_seqlens
and states stored as S ([.., V, K]) instead of h = S^T.  Both change only
addressing, so every path must give the same bits as the default layout,
whose results the parity tests hold against the oracle.  All calls go
through the C ABI."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS
LENS = [1, 63, 64, 65, 130, 7, 0, 200]

CASES = {
    # (workload, overrides, n_segments, force_path)
    "tc_serial": (W["wide_varlen_bf16"], dict(H=2), 1, 2),
    "tc_split": (W["wide_varlen_bf16"], dict(H=2, with_h0=True), 4, 2),
    "simt_split_f32": (W["wide_varlen_bf16"], dict(H=2, dtype="f32", with_h0=True), 2, 1),
    "beta_free_split": (W["gla_k256_v512_bf16"], dict(K=128, V=256, H=2), 2, 2),
}


def run(x, cu, n_segments, force_path, state_layout="kv"):
    d = to_dev(x)
    h0 = d["h0"]
    if h0 is not None and state_layout == "vk":
        h0 = h0.transpose(-1, -2).contiguous()
    o, ht = pkg.gdr_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=cu, h0=h0,
                              n_segments=n_segments, force_path=force_path,
                              state_layout=state_layout)
    torch.cuda.synchronize()
    if state_layout == "vk":
        ht = ht.transpose(-1, -2)
    return o, ht


@pytest.mark.parametrize("case", sorted(CASES))
def test_int64_seqlens_give_the_same_bits(case):
    w, over, S, path = CASES[case]
    x = synthetic.make_inputs(synthetic.small(w, **over), lengths=LENS)
    cu32 = x["cu_seqlens"].cuda()
    o1, h1 = run(x, cu32, S, path)
    o2, h2 = run(x, cu32.to(torch.int64), S, path)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("case", sorted(CASES))
def test_states_as_s_give_the_same_bits(case):
    w, over, S, path = CASES[case]
    x = synthetic.make_inputs(synthetic.small(w, **over), lengths=LENS)
    cu = x["cu_seqlens"].cuda()
    o1, h1 = run(x, cu, S, path)
    o2, h2 = run(x, cu, S, path, state_layout="vk")
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_dense_layout_states_as_s():
    w = synthetic.small(W["tiny_dense_f32"], T=130, H=2, B=3)
    x = synthetic.make_inputs(w)
    o1, h1 = run(x, None, 1, 0)
    o2, h2 = run(x, None, 1, 0, state_layout="vk")
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("state_layout", ["kv", "vk"])
def test_recurrent_with_both_flags(state_layout):
    w = synthetic.small(W["decode_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=[1, 4, 0, 2, 3])
    pool, idx = synthetic.make_state_pool(x, 9)
    d = to_dev(x)
    outs = []
    for cu in (d["cu_seqlens"], d["cu_seqlens"].to(torch.int64)):
        p = pool.clone().cuda()
        if state_layout == "vk":
            p = p.transpose(-1, -2).contiguous()
        o = pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=cu,
                                  state=p, state_indices=idx.cuda(), state_layout=state_layout)
        torch.cuda.synchronize()
        outs.append((o, p.transpose(-1, -2) if state_layout == "vk" else p))
    ref_p = pool.clone().cuda()
    ref_o = pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  cu_seqlens=d["cu_seqlens"], state=ref_p,
                                  state_indices=idx.cuda())
    torch.cuda.synchronize()
    for o, p in outs:
        assert torch.equal(o, ref_o) and torch.equal(p, ref_p)


def test_host_entry_with_int64_seqlens():
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=LENS)
    o1, h1 = run(x, x["cu_seqlens"].cuda(), 0, 0)
    o2, h2 = pkg.gdr_chunk_fwd_host(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                    cu_seqlens=x["cu_seqlens"].to(torch.int64))
    assert torch.equal(o1.cpu(), o2) and torch.equal(h1.cpu(), h2)
