"""GPU parity of the CUDA path against the FP64 oracle, element by element,
at sizes the oracle finishes in seconds (several chunks, ragged tails, empty
sequences), plus the launch-plan and run-to-run bit identity, graph capture,
NaN-poisoned outputs, the device status word, the host-buffer entry point
and caller-provided workspace.  All calls go through the C ABI."""
import math

import numpy as np
import pytest
import torch

from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import (TOL_BF16, TOL_F32, assert_parity, rel_l2_masked, run_gpu, run_oracle,
                      to_dev, tol_of)

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS


def poisoned_outputs(x):
    """o and ht filled with NaN, so an element the library leaves unwritten
    fails the comparison (a fresh allocation may hold an earlier result)."""
    n = x["N"] if x["cu_seqlens"] is not None else x["B"]
    o = torch.full(x["v"].shape, float("nan"), dtype=x["v"].dtype, device="cuda")
    ht = torch.full((n, x["H"], x["K"], x["V"]), float("nan"), dtype=torch.float32,
                    device="cuda")
    return o, ht


def check(x, tol=None, **kw):
    tol = tol or tol_of(x)
    o0, ht0 = poisoned_outputs(x)
    o, ht = run_gpu(x, o=o0, ht=ht0, **kw)
    ro, rht = run_oracle(x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    eo, eh, _, _ = assert_parity(x, o, ht, ro, rht, tol, label=str(kw))
    return eo, eh


@pytest.mark.parametrize("S", [1, 2, 4])
def test_tiny_dense_f32(S):
    """FP32 tiny dense workload (B=1, T=256, H=2, K=V=64, h0 in, ht out)."""
    check(synthetic.make_inputs(W["tiny_dense_f32"]), n_segments=S)


@pytest.mark.parametrize("K,V", [(16, 16), (32, 64), (128, 32), (256, 128)])
def test_f32_shapes(K, V):
    w = synthetic.small(W["tiny_dense_f32"], K=K, V=V, T=200, H=2, B=2)
    check(synthetic.make_inputs(w))


RAGGED = [1, 63, 64, 65, 127, 128, 257, 7, 300]
# 1: CUDA-core FP32 path; 2: tensor-core path (BF16, K = V = 128, delta rule)
PATHS = [1, 2]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("S", [1, 2, 4, 16])
def test_bf16_ragged_varlen(S, path):
    w = synthetic.small(W["wide_varlen_bf16"], H=3)
    check(synthetic.make_inputs(w, lengths=RAGGED), n_segments=S, force_path=path)


@pytest.mark.parametrize("path", PATHS)
def test_bf16_varlen_with_empty_sequences_and_h0(path):
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    x = synthetic.make_inputs(w, lengths=[0, 70, 0, 129, 0])
    o0, ht0 = poisoned_outputs(x)
    o, ht = run_gpu(x, force_path=path, o=o0, ht=ht0)
    ro, rht = run_oracle(x)
    assert_parity(x, o, ht, ro, rht, TOL_BF16, label=f"empty sequences, path {path}")
    # an empty sequence hands back its initial state exactly
    assert torch.equal(ht[0].cpu(), x["h0"][0])
    assert torch.equal(ht[4].cpu(), x["h0"][4])


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8, 16])
def test_bf16_dense_h0_segments(S, path):
    w = synthetic.small(W["long_16k_bf16"], B=2, T=1000, H=2, with_h0=True)
    check(synthetic.make_inputs(w), n_segments=S, force_path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("S", [1, 4])
def test_beta_free_k256_v512(S, path):
    w = synthetic.small(W["gla_k256_v512_bf16"], T=300, H=2)
    check(synthetic.make_inputs(w), n_segments=S, force_path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("S", [1, 3])
def test_beta_free_k128_v256_varlen(S, path):
    w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=3)
    check(synthetic.make_inputs(w, lengths=[1, 64, 65, 200, 0, 130]), n_segments=S,
          force_path=path)


@pytest.mark.parametrize("path", PATHS)
def test_beta_free_one_chunk_per_segment(path):
    """n_segments at or above the chunk count: every chunk its own segment,
    the chunk-parallel producer dataflow (per-chunk FP32 contributions, the
    ordered scalar-decay scan, each chunk's output from its boundary
    state)."""
    w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=2, with_h0=True)
    check(synthetic.make_inputs(w, lengths=[1, 64, 65, 700, 0, 300]), n_segments=4096,
          force_path=path)


def many_lengths(n, hi, seed):
    """Seeded sequence lengths in [0, hi], zeros included."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, hi + 1, (n,), generator=g).tolist()


@pytest.mark.parametrize("S", [1, 4])
def test_many_short_sequences_delta(S):
    """600 sequences of 0-200 tokens: every persistent CTA walks several
    chains, the chain hand-over ring wraps many times, most chunks are ragged."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    check(synthetic.make_inputs(w, lengths=many_lengths(600, 200, 11)), n_segments=S,
          force_path=2)


@pytest.mark.parametrize("S", [8, 16])
def test_common_segment_length(S):
    """One segment length for every sequence, ceil(longest / S) chunks: the
    long sequence is split; sequences of exactly that length or shorter
    (empty, one token, ragged) run whole in the output pass from h0 to ht;
    one a token longer is split into a full segment and a one-token one."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    per = -(-47 // S)  # 3000 tokens: 47 chunks
    lens = [3000, 64 * per, 64 * per + 1, 0, 1, 200]
    check(synthetic.make_inputs(w, lengths=lens), n_segments=S, force_path=2)


@pytest.mark.parametrize("S", [4, 16])
def test_common_segment_length_beta_free(S):
    """The beta-free mode at one segment length for every sequence: the long
    sequence is split into ceil(40 / S)-chunk runs (two 128-column value
    tiles, K = 128); shorter ones, an empty one and one of exactly that
    length run whole in the output pass from h0 to ht."""
    w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=2, with_h0=True)
    per = -(-40 // S)  # 2540 tokens: 40 chunks
    lens = [2540, 64 * per, 64 * per + 1, 0, 1, 90]
    check(synthetic.make_inputs(w, lengths=lens), n_segments=S, force_path=2)


@pytest.mark.parametrize("case", ["two_long", "default_plan"])
def test_common_segment_length_long_sequences(case):
    """Two sequences of 127 chunks or more (the sequence order's top bucket,
    where it does not rank them): the segment length follows the longer one
    (201 chunks, 26 a segment at S = 8), the other splits into 5; a
    sequence of exactly 26 chunks runs whole.  Then a skewed batch at the
    default plan, which splits the long sequence only."""
    w = synthetic.small(W["wide_varlen_bf16"], H=1, with_h0=True)
    if case == "two_long":
        lens = [130 * 64 - 5, 200 * 64 + 7, 300, 0, 64 * 26]
        check(synthetic.make_inputs(w, lengths=lens), n_segments=8, force_path=2)
    else:
        w = synthetic.small(W["skewed_varlen_h4_bf16"], H=2, with_h0=True)
        lens = [8192] + [128 + 37 * i for i in range(12)]
        x = synthetic.make_inputs(w, lengths=lens)
        import chunked_gated_delta_rule_gb300 as pkg
        assert pkg.gdr_plan_query(1, sum(lens), 2, 128, 128, N=len(lens), dtype=1,
                                  max_len=8192)["n_segments"] > 1
        check(x)


@pytest.mark.parametrize("S", [2, 8])
def test_segment_prescan_both_kernels(S):
    """Multi-chunk ragged segments, an empty sequence: at 4 heads, S = 2 runs
    each summary (c_s, M_s) as its own chain; S = 8 has too many segments for
    one wave and runs both summaries of a segment in one CTA."""
    w = synthetic.small(W["wide_varlen_bf16"], H=4)
    check(synthetic.make_inputs(w, lengths=[1000, 700, 64, 0, 333]), n_segments=S,
          force_path=2)


@pytest.mark.parametrize("S", [1, 2])
def test_many_short_sequences_beta_free(S):
    w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=2)
    check(synthetic.make_inputs(w, lengths=many_lengths(300, 200, 12)), n_segments=S,
          force_path=2)


@pytest.mark.parametrize("path", PATHS)
def test_literal_beta_zero(path):
    """An all-zero beta tensor freezes the state: o_t = e^{G_t} h0^T q_t / sqrt(K)."""
    w = synthetic.small(W["long_16k_bf16"], T=200, H=2, with_h0=True)
    x = synthetic.make_inputs(w, beta_zero=True)
    check(x, force_path=path)
    check(x, n_segments=2, force_path=path)


def test_scale_override():
    x = synthetic.make_inputs(synthetic.small(W["tiny_dense_f32"], T=130))
    o1, _ = run_gpu(x)
    o2, _ = run_gpu(x, scale=0.5)
    s = 1 / math.sqrt(x["K"])
    torch.testing.assert_close(o2, o1 * (0.5 / s), rtol=1e-5, atol=1e-6)


# --------------------------------------------------------------------------
# bit identity, graph capture, poisoning, status, host entry, workspace
# --------------------------------------------------------------------------
def _bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu()


@pytest.mark.parametrize("S", [1, 4])
def test_bit_identical_across_plans_and_repeats(S):
    """CUDA-core path: every value-tile width gives the same bits; the
    tensor-core path (one plan per shape) gives the same bits run to run."""
    w = synthetic.small(W["wide_varlen_bf16"], H=2)
    x = synthetic.make_inputs(w, lengths=RAGGED)
    ref_o, ref_h = run_gpu(x, n_segments=S, force_path=1, force_bv=64)
    for bv in (16, 32, 64, 64):
        o, ht = run_gpu(x, n_segments=S, force_path=1, force_bv=bv)
        assert torch.equal(_bits(o), _bits(ref_o)), bv
        assert torch.equal(_bits(ht), _bits(ref_h)), bv
    tc_o, tc_h = run_gpu(x, n_segments=S, force_path=2)
    for _ in range(3):
        o, ht = run_gpu(x, n_segments=S, force_path=2)
        assert torch.equal(_bits(o), _bits(tc_o))
        assert torch.equal(_bits(ht), _bits(tc_h))


@pytest.mark.parametrize("case", ["two_level_h0", "two_level_no_ht", "two_level_varlen",
                                  "single_many_heads"])
def test_tensor_core_composition(case):
    """The segment composition on the tensor cores (FP32 operands carried as
    BF16 hi + lo pairs): its two-level form (one head, 64 one-chunk segments
    in groups of 8) from h0, the same without the final state (the last
    group step is skipped), over sequences with different segment counts
    (empty, one chunk, ragged, a partial last group); its single ordered pass
    at 16 heads.  Element by element against the FP64 oracle."""
    if case == "single_many_heads":
        w = synthetic.small(W["long_16k_bf16"], T=1024, H=16, with_h0=True)
        x, S = synthetic.make_inputs(w), 9
    elif case == "two_level_varlen":
        w = synthetic.small(W["wide_varlen_bf16"], H=1, with_h0=True)
        x, S = synthetic.make_inputs(w, lengths=[4096, 0, 64, 1000, 3000]), 64
    else:
        w = synthetic.small(W["long_16k_bf16"], T=4096, H=1, with_h0=True)
        x, S = synthetic.make_inputs(w), 64
    if case != "two_level_no_ht":
        check(x, n_segments=S, force_path=2)
        return
    o0, _ = poisoned_outputs(x)
    o, ht = run_gpu(x, o=o0, n_segments=S, force_path=2, output_final_state=False)
    assert ht is None and torch.isfinite(o.float()).all()
    ro, _ = run_oracle(x)
    assert rel_l2_masked(o, ro) <= tol_of(x)


@pytest.mark.parametrize("case", ["delta_serial", "delta_split_chains", "delta_split_dual",
                                  "delta_two_level", "beta_free_split", "beta_free_k256"])
def test_tensor_core_bits_identical_across_grids(case):
    """Bit-identical across launch configurations: the persistent
    tensor-core kernels (preparation, scan, both pre-scans, the composition
    in one and two levels, the beta-free scan) with 1, 5 and 37 CTAs give the
    bits of their one-CTA-per-SM grids
    (every chain and chunk is computed by one CTA in a fixed order whichever
    CTA pulls it)."""
    if case == "delta_two_level":  # the two-level tensor-core composition
        w = synthetic.small(W["long_16k_bf16"], T=4096, H=1, with_h0=True)
        lens, S = None, 64
    elif case.startswith("delta"):
        w = synthetic.small(W["wide_varlen_bf16"], H=4)
        lens = [1000, 700, 64, 0, 333] if case != "delta_serial" else RAGGED
        S = {"delta_serial": 1, "delta_split_chains": 2, "delta_split_dual": 8}[case]
    elif case == "beta_free_split":
        w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=3)
        lens, S = [1, 64, 65, 200, 0, 130, 700], 3
    else:
        w = synthetic.small(W["gla_k256_v512_bf16"], T=600, H=2)
        lens, S = None, 2
    x = synthetic.make_inputs(w, lengths=lens)
    ref_o, ref_h = run_gpu(x, n_segments=S, force_path=2)
    for limit in (1, 5, 37):
        o, ht = run_gpu(x, n_segments=S, force_path=2, grid_limit=limit)
        assert torch.equal(_bits(o), _bits(ref_o)), (case, limit)
        assert torch.equal(_bits(ht), _bits(ref_h)), (case, limit)


def test_graph_capture_matches_eager():
    import chunked_gated_delta_rule_gb300 as pkg
    x = to_dev(synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=2),
                                     lengths=RAGGED))
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"])
    o_e, ht_e = pkg.gdr_chunk_fwd(*args, cu_seqlens=x["cu_seqlens"])
    o = torch.full_like(o_e, float("nan"))
    ht = torch.full_like(ht_e, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        pkg.gdr_chunk_fwd(*args, cu_seqlens=x["cu_seqlens"], o=o, ht=ht)  # warm-up
        torch.cuda.synchronize()
        o.fill_(float("nan"))
        with torch.cuda.graph(graph, stream=s):
            pkg.gdr_chunk_fwd(*args, cu_seqlens=x["cu_seqlens"], o=o, ht=ht)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(o), _bits(o_e))
    assert torch.equal(_bits(ht), _bits(ht_e))


def test_nan_poisoned_outputs_are_fully_written():
    import chunked_gated_delta_rule_gb300 as pkg
    x = to_dev(synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=2),
                                     lengths=RAGGED))
    o = torch.full(x["v"].shape, float("nan"), dtype=x["v"].dtype, device="cuda")
    ht = torch.full((len(RAGGED), 2, 128, 128), float("nan"), device="cuda")
    pkg.gdr_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=x["cu_seqlens"],
                      o=o, ht=ht)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert torch.isfinite(ht).all()


def test_status_word_reports_malformed_cu_seqlens():
    import chunked_gated_delta_rule_gb300 as pkg
    x = to_dev(synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=1),
                                     lengths=[64, 64, 64]))
    cu = torch.tensor([0, 100, 50, 192], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full(x["v"].shape, 7.0, dtype=x["v"].dtype, device="cuda")
    pkg.gdr_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_seqlens=cu, o=o,
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -5
    assert bool((o == 7.0).all())  # nothing computed


def test_host_entry_matches_device_entry():
    import chunked_gated_delta_rule_gb300 as pkg
    x = synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=2), lengths=RAGGED)
    o_d, ht_d = run_gpu(x)
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
    o_h, ht_h = pkg.gdr_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                       cu_seqlens=pin["cu_seqlens"])
    assert torch.equal(_bits(o_h), _bits(o_d))
    assert torch.equal(_bits(ht_h), _bits(ht_d))


def _host_run(x, **kw):
    import chunked_gated_delta_rule_gb300 as pkg
    pin = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()}
    return pkg.gdr_chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"],
                                  cu_seqlens=pin["cu_seqlens"], h0=pin["h0"], **kw)


@pytest.mark.parametrize("case", ["wide_varlen", "dense_h0", "one_sequence", "one_varlen_f32"])
def test_host_entry_groups_match_device_entry(case):
    """Inputs of 48 MB and more are cut into groups whose copies overlap the
    passes: groups of whole sequences, or pieces of one long sequence run as
    consecutive passes with the state carried on the device.  With the plan
    pinned (one segment) every result is bit-identical to the one-call
    device entry (the serial chain hands its FP32 state across a piece
    boundary unchanged)."""
    if case == "wide_varlen":  # 130 MB in: 4 groups of whole sequences
        x = synthetic.make_inputs(W["wide_varlen_bf16"])
    elif case == "dense_h0":  # 8 rows x 4096 tokens x 4 heads with h0: 3 groups of batch rows
        x = synthetic.make_inputs(synthetic.small(W["long_16k_bf16"], B=8, T=4096, H=4,
                                                  with_h0=True))
    elif case == "one_sequence":  # 1 row x 16K tokens x 4 heads, h0: 2 pieces
        x = synthetic.make_inputs(synthetic.small(W["long_16k_bf16"], H=4, with_h0=True))
    else:  # one varlen sequence, FP32 (the CUDA-core path), 3 pieces, ragged end
        x = synthetic.make_inputs(synthetic.small(W["tiny_dense_f32"], H=4, K=128, V=128),
                                  lengths=[20000 + 37])
    o_d, ht_d = run_gpu(x, n_segments=1)
    o_h, ht_h = _host_run(x, n_segments=1)
    assert torch.equal(_bits(o_h), _bits(o_d.cpu()))
    assert torch.equal(_bits(ht_h), _bits(ht_d.cpu()))


def test_default_plan_uses_tensor_core_path_for_bf16_k128():
    import chunked_gated_delta_rule_gb300 as pkg
    assert pkg.gdr_plan_query(1, 10456, 16, 128, 128, N=32)["path"] == 2
    assert pkg.gdr_plan_query(1, 256, 2, 64, 64, dtype=0)["path"] == 1
    assert pkg.gdr_plan_query(2, 8192, 4, 256, 512, beta_free=True)["path"] == 2
    assert pkg.gdr_plan_query(2, 8192, 4, 64, 512, beta_free=True)["path"] == 1


def test_caller_workspace_matches_internal_allocation():
    import chunked_gated_delta_rule_gb300 as pkg
    x = synthetic.make_inputs(synthetic.small(W["wide_varlen_bf16"], H=2), lengths=RAGGED)
    o_a, ht_a = run_gpu(x, n_segments=2)
    nbytes = pkg.gdr_workspace_size(1, x["T"], 2, 128, 128, N=len(RAGGED), n_segments=2)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o_b, ht_b = run_gpu(x, n_segments=2, workspace=ws)
    assert torch.equal(_bits(o_a), _bits(o_b))
    assert torch.equal(_bits(ht_a), _bits(ht_b))
    with pytest.raises(pkg.GdrError):
        run_gpu(x, n_segments=2, workspace=ws[: nbytes // 2])
