"""gdr_chunk_fwd_noalloc: the entry point that allocates nothing (its scratch
is a fixed 64 MiB array inside the library), for callers that must not
allocate device memory during a call.  Collected last on purpose, so a run
that stops at the first failure has run every other test before it.

Checks, through the C ABI: two calls in a row each match gdr_chunk_fwd (the
shared scratch keeps the previous call's contents, which must not leak into
the next result), and a problem that needs more scratch than the array holds
is refused before any work."""
import ctypes

import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import api, synthetic
from gpu_util import TOL_BF16, TOL_F32, rel_l2_masked, to_dev

W = synthetic.WORKLOADS


def _cases():
    yield "tiny_dense_f32", synthetic.make_inputs(W["tiny_dense_f32"]), 1, TOL_F32
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    yield "ragged_varlen_bf16", synthetic.make_inputs(w, lengths=[1, 63, 64, 65, 200]), 1, TOL_BF16
    w = synthetic.small(W["long_16k_bf16"], T=700, H=2)
    yield "dense_bf16_segments", synthetic.make_inputs(w), 4, TOL_BF16


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_on_two_calls_in_a_row():
    for name, x, S, tol in _cases():
        d = to_dev(x)
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
        kw = dict(cu_seqlens=d["cu_seqlens"], h0=d["h0"], n_segments=S)
        o_ref, ht_ref = pkg.gdr_chunk_fwd(*args, **kw)
        torch.cuda.synchronize()
        o_ref64 = o_ref.double().cpu().numpy()
        ht_ref64 = ht_ref.double().cpu().numpy()
        for call in range(2):
            o = torch.full_like(o_ref, float("nan"))
            ht = torch.full_like(ht_ref, float("nan"))
            pkg.gdr_chunk_fwd_noalloc(*args, o=o, ht=ht, **kw)
            torch.cuda.synchronize()
            eo, eh = rel_l2_masked(o, o_ref64), rel_l2_masked(ht, ht_ref64)
            assert eo <= tol and eh <= tol, (name, call, eo, eh)


def test_noalloc_refuses_problems_larger_than_its_scratch():
    """Refused on the host before any CUDA call (runs without a GPU)."""
    lib = pkg.load_library()
    # FP32 inputs run on the CUDA-core path, which keeps per-chunk W, U,
    # h_pre and v_new in scratch: this size needs far more than 64 MiB
    dims = api.make_dims(1, 16384, 16, 64, 64, dtype=api.GDR_F32)
    assert (pkg.gdr_workspace_size(1, 16384, 16, 64, 64, dtype=api.GDR_F32)
            > api.NOALLOC_SCRATCH_BYTES)
    p = ctypes.c_void_p(0x1000)
    rc = lib.gdr_chunk_fwd_noalloc(ctypes.byref(dims), p, p, p, p, p, None, None, p, p, 0, None)
    assert rc == -6
    bad = api.make_dims(1, 128, 2, 60, 64)
    rc = lib.gdr_chunk_fwd_noalloc(ctypes.byref(bad), p, p, p, p, p, None, None, p, p, 0, None)
    assert rc == -1
