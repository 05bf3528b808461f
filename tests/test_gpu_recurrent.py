"""GPU parity of gdr_recurrent_fwd (the per-token recurrence on rows of a
state pool) against the FP64 oracle: each sequence's pool row is its h0 and
must end as the oracle's ht; rows no sequence names stay bit-identical.  All
calls go through the C ABI."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import TOL_BF16, TOL_F32, assert_parity, rel_l2_masked, run_oracle, to_dev

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS


def run_pool(x, n_states, use_indices=True, seed=1):
    pool, idx = synthetic.make_state_pool(x, n_states, seed)
    if not use_indices:  # row n for sequence n
        idx = torch.arange(x["N"], dtype=torch.int32)
        if x["h0"] is not None:
            pool[: x["N"]] = x["h0"]
    d = to_dev(x)
    dpool = pool.cuda()
    o = torch.full(d["v"].shape, float("nan"), dtype=d["v"].dtype, device="cuda")
    pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                          state=dpool, state_indices=idx.cuda() if use_indices else None, o=o)
    torch.cuda.synchronize()
    return o, dpool.cpu(), pool, idx


def check(x, n_states, tol_o, tol_h, **kw):
    o, after, before, idx = run_pool(x, n_states, **kw)
    ro, rht = run_oracle(x)
    assert torch.isfinite(o.float()).all()
    eo, eh, _, _ = assert_parity(x, o, after[idx.long()], ro, rht, tol_o, tol_h, label="recurrent")
    untouched = torch.ones(n_states, dtype=torch.bool)
    untouched[idx.long()] = False
    assert torch.equal(after[untouched], before[untouched])
    return eo, eh


def test_decode_one_token_per_sequence_bf16():
    """The decode workload's shape at 64 sequences: one token each."""
    w = synthetic.small(W["decode_bf16"], n_seqs=64)
    x = synthetic.make_inputs(w)
    # o is BF16 (one rounding); the state is FP32 arithmetic on the same inputs
    check(x, 160, TOL_BF16, 1e-5)


@pytest.mark.parametrize("delta", [True, False])
def test_few_tokens_per_sequence_varlen_bf16(delta):
    """Rows of 0-9 tokens (a sequence without tokens keeps its state)."""
    w = synthetic.small(W["decode_bf16"], H=4, delta=delta)
    lens = [1, 3, 0, 9, 2, 5, 1, 7, 4, 0, 6, 8]
    x = synthetic.make_inputs(w, lengths=lens)
    check(x, 40, TOL_BF16, 1e-5)


@pytest.mark.parametrize("K,V", [(64, 64), (128, 96), (256, 128), (32, 512)])
def test_shapes_f32(K, V):
    w = synthetic.small(W["tiny_dense_f32"], K=K, V=V, T=5, H=2, B=3)
    x = synthetic.make_inputs(w)
    check(x, 7, TOL_F32, TOL_F32)


def test_rows_by_sequence_number_dense():
    w = synthetic.small(W["tiny_dense_f32"], T=3, H=2, B=4)
    x = synthetic.make_inputs(w)
    check(x, 4, TOL_F32, TOL_F32, use_indices=False)


def test_chained_steps_equal_the_chunked_forward():
    """Token after token through gdr_recurrent_fwd equals one gdr_chunk_fwd
    over the whole sequences (both against the oracle, and each other)."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, dtype="f32")
    x = synthetic.make_inputs(w, lengths=[70, 5, 130])
    ro, rht = run_oracle(x)
    d = to_dev(x)
    cu = x["cu_seqlens"].tolist()
    N = x["N"]
    pool = torch.zeros(N, x["H"], x["K"], x["V"], device="cuda")
    o = torch.full(d["v"].shape, float("nan"), device="cuda")
    for step in range(max(cu[i + 1] - cu[i] for i in range(N))):
        rows = [n for n in range(N) if cu[n] + step < cu[n + 1]]
        sel = torch.tensor([cu[n] + step for n in rows])
        one = torch.arange(len(rows) + 1, dtype=torch.int32).cuda()
        ostep = torch.empty(1, len(rows), x["H"], x["V"], device="cuda")
        pkg.gdr_recurrent_fwd(d["q"][:, sel].contiguous(), d["k"][:, sel].contiguous(),
                              d["v"][:, sel].contiguous(), d["g"][:, sel].contiguous(),
                              d["beta"][:, sel].contiguous(), cu_seqlens=one, state=pool,
                              state_indices=torch.tensor(rows, dtype=torch.int32).cuda(),
                              o=ostep)
        o[:, sel] = ostep
    torch.cuda.synchronize()
    assert_parity(x, o, pool, ro, rht, TOL_F32, label="chained decode steps")
    oc, htc = pkg.gdr_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert rel_l2_masked(o, oc.cpu().double().numpy()) <= 2 * TOL_F32


def test_out_of_range_index_reports_and_skips():
    w = synthetic.small(W["decode_bf16"], n_seqs=3, H=2)
    x = synthetic.make_inputs(w)
    d = to_dev(x)
    pool = torch.randn(5, 2, 128, 128, device="cuda")
    before = pool.clone()
    idx = torch.tensor([0, 9, 2], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full(d["v"].shape, float("nan"), dtype=d["v"].dtype, device="cuda")
    pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"],
                          state=pool, state_indices=idx, o=o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -7  # GDR_ERR_INDEX
    assert torch.isnan(o[0, 1].float()).all()          # sequence 1 skipped
    assert torch.isfinite(o[0, [0, 2]].float()).all()  # the others computed
    assert torch.equal(pool[[1, 3, 4]], before[[1, 3, 4]])
