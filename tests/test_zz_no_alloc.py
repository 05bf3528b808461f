"""gdr_chunk_fwd_noalloc: the forward pass that allocates no device memory.

Some callers cannot let a library allocate GPU memory while they run: serving
engines that reserve nearly all of HBM for their caches at start-up and treat
a later allocation as a failure, frameworks that own the allocator, code
where an allocation call is not allowed.  This entry point takes its scratch
from a fixed 64 MiB array inside the library instead.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test.

Checks, through the C ABI:
  * consecutive calls on different inputs (so scratch left by one call could
    change the next one's result) each give exactly the bits of
    gdr_chunk_fwd on the same inputs: both run the same kernels with the
    same plan, so nothing but a fault in the scratch handling can differ;
  * misaligned q, k, v, o (the CUDA-core path, which needs more scratch than
    the tensor-core path it replaces) run and match too;
  * device free memory is the same before and after the calls;
  * a problem that needs more scratch than the array holds is refused before
    any work, and invalid or unsupported arguments return the codes
    gdr_chunk_fwd returns.
"""
import ctypes

import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import api, synthetic
from gpu_util import to_dev

W = synthetic.WORKLOADS


def _cases():
    """(name, inputs, n_segments): both paths, dense and varlen, serial and
    split, delta rule and beta-free, with and without h0."""
    yield "tiny_dense_f32", synthetic.make_inputs(W["tiny_dense_f32"]), 1
    w = synthetic.small(W["wide_varlen_bf16"], H=2, with_h0=True)
    yield "ragged_varlen_bf16", synthetic.make_inputs(w, lengths=[1, 63, 64, 65, 200]), 1
    w = synthetic.small(W["long_16k_bf16"], T=700, H=2, seed=3)
    yield "dense_bf16_segments", synthetic.make_inputs(w), 4
    w = synthetic.small(W["gla_k256_v512_bf16"], B=1, T=300, H=2, K=128, V=128, seed=5)
    yield "beta_free_bf16", synthetic.make_inputs(w), 2


def _misaligned(t):
    """A copy of t whose data starts 2 bytes past a 16-byte boundary."""
    flat = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    view = flat[1:1 + t.numel()].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 16 != 0
    return view


def _bits_equal(a, b):
    ints = {1: torch.int8, 2: torch.int16, 4: torch.int32}
    return (a.shape == b.shape and a.dtype == b.dtype
            and torch.equal(a.view(ints[a.element_size()]), b.view(ints[b.element_size()])))


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_bit_for_bit_on_consecutive_calls():
    runs = []
    for name, x, S in _cases():
        d = to_dev(x)
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
        kw = dict(cu_seqlens=d["cu_seqlens"], h0=d["h0"], n_segments=S)
        o_ref, ht_ref = pkg.gdr_chunk_fwd(*args, **kw)
        runs.append((name, args, kw, o_ref, ht_ref))
    # misaligned q, k, v, o: the same shape moves to the CUDA-core path
    w = synthetic.small(W["wide_varlen_bf16"], H=2, seed=9)
    d = to_dev(synthetic.make_inputs(w, lengths=[70, 129]))
    args = (_misaligned(d["q"]), _misaligned(d["k"]), _misaligned(d["v"]), d["g"], d["beta"])
    o_mis = _misaligned(torch.zeros_like(d["v"]))
    kw = dict(cu_seqlens=d["cu_seqlens"], h0=None, n_segments=0)
    o_ref, ht_ref = pkg.gdr_chunk_fwd(*args, **kw)
    runs.append(("misaligned_varlen_bf16", args, dict(kw, o=o_mis), o_ref, ht_ref))
    torch.cuda.synchronize()

    # every case in turn, then the first again: each call follows one on
    # other inputs and shapes.  Outputs of every call are allocated (and
    # NaN-filled once, so that the fill kernels are loaded) up front, and the
    # results are compared only after the last call: a comparison allocates
    # torch temporaries, which would move the free-memory reading.
    order = list(range(len(runs))) + [0]
    outs = []
    for i in order:
        _, _, kw, o_ref, ht_ref = runs[i]
        o = kw.get("o") if i == len(runs) - 1 else None
        outs.append((o if o is not None else torch.empty_like(o_ref), torch.empty_like(ht_ref)))
        for t in outs[-1]:
            t.fill_(float("nan"))
    # one call first, which looks up the scratch array's device address
    name, args, kw, o_ref, ht_ref = runs[0]
    pkg.gdr_chunk_fwd_noalloc(*args, **{**kw, "o": torch.empty_like(o_ref),
                                        "ht": torch.empty_like(ht_ref)})
    torch.cuda.synchronize()
    pkg.gdr_release_cached()  # the allocating entry's pooled scratch goes back
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for j, i in enumerate(order):
        name, args, kw, _, _ = runs[i]
        o, ht = outs[j]
        pkg.gdr_chunk_fwd_noalloc(*args, **{**kw, "o": o, "ht": ht})
        torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    for j, i in enumerate(order):
        name, _, _, o_ref, ht_ref = runs[i]
        assert _bits_equal(outs[j][0], o_ref), (name, j, "o")
        assert _bits_equal(outs[j][1], ht_ref), (name, j, "ht")
    assert free_after == free_before, (free_before, free_after)


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
    # the codes gdr_chunk_fwd returns: K not a multiple of 16 is unsupported,
    # a missing q or a segment count below zero invalid, above 64 unsupported
    bad = api.make_dims(1, 128, 2, 60, 64)
    for entry in (lib.gdr_chunk_fwd_noalloc, lib.gdr_chunk_fwd):
        assert entry(ctypes.byref(bad), p, p, p, p, p, None, None, p, p, 0, None) == -2
    ok = api.make_dims(1, 128, 2, 64, 64)
    assert lib.gdr_chunk_fwd_noalloc(ctypes.byref(ok), None, p, p, p, p, None, None, p, p, 0,
                                     None) == -1
    assert lib.gdr_chunk_fwd_noalloc(ctypes.byref(ok), p, p, p, p, p, None, None, p, p, -1,
                                     None) == -1
    assert lib.gdr_chunk_fwd_noalloc(ctypes.byref(ok), p, p, p, p, p, None, None, p, p, 65,
                                     None) == -2
