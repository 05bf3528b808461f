"""The C-ABI library on the CPU: it loads, exports every symbol the header
declares, and its host-only logic (argument checks, plan, workspace size,
error strings) works without a GPU.  No compute call is made."""
import ctypes
import os
import re

import pytest

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_delta_rule_gb300 import build
    build.build()
    return pkg.load_library()


def declared_functions(paths=None):
    names = set()
    for path in paths or HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"\b(gdr_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_expected_entry_points():
    assert declared_functions([HEADER]) == sorted(api.EXPORTS)
    assert declared_functions() == sorted(api.EXPORTS + api.SELFTEST_EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert callable(getattr(lib, name))


def test_version_and_error_strings(lib):
    assert pkg.gdr_version() == 100
    assert pkg.gdr_error_string(0) == "ok"
    assert pkg.gdr_error_string(-5) == "malformed cu_seqlens"
    assert pkg.gdr_error_string(12345) == "unknown error code"


def _fwd(lib, dims, q=1, k=1, v=1, g=1, o=1, cu=None, n_segments=0, opt=None):
    p = lambda x: None if x is None else ctypes.c_void_p(0x1000 * x)
    if opt is None:
        return lib.gdr_chunk_fwd(ctypes.byref(dims), p(q), p(k), p(v), p(g), None, p(cu),
                                 None, p(o), None, n_segments, None)
    return lib.gdr_chunk_fwd_ex(ctypes.byref(dims), p(q), p(k), p(v), p(g), None, p(cu),
                                None, p(o), None, n_segments, ctypes.byref(opt), None)


def test_argument_checks_reject_before_any_gpu_work(lib):
    ok = api.make_dims(1, 128, 2, 64, 64)
    assert _fwd(lib, ok, q=None) == -1
    assert _fwd(lib, ok, o=None) == -1
    assert _fwd(lib, api.make_dims(1, 128, 2, 64, 64, dtype=7)) == -1
    assert _fwd(lib, api.make_dims(0, 128, 2, 64, 64)) == -1
    assert _fwd(lib, api.make_dims(1, -1, 2, 64, 64)) == -1
    assert _fwd(lib, api.make_dims(1, 128, 2, 60, 64)) == -2      # K % 16
    assert _fwd(lib, api.make_dims(1, 128, 2, 512, 64)) == -2     # K > 256
    assert _fwd(lib, api.make_dims(1, 128, 2, 64, 2048)) == -2    # V > 1024
    assert _fwd(lib, api.make_dims(2, 128, 2, 64, 64, N=3), cu=5) == -1  # varlen needs B == 1
    assert _fwd(lib, api.make_dims(1, 128, 2, 64, 64, N=3), cu=None) == -1  # N>0 needs cu
    assert _fwd(lib, ok, cu=5) == -1                                # cu given, N == 0
    assert _fwd(lib, ok, n_segments=-1) == -1
    # at most 4096 segments in the beta-free mode (beta NULL, as here), 64
    # for the delta rule (the plan query needs no pointers)
    assert _fwd(lib, ok, n_segments=4097) == -2
    with pytest.raises(pkg.GdrError):
        pkg.gdr_plan_query(1, 128, 2, 64, 64, n_segments=65)
    assert pkg.gdr_plan_query(1, 128, 2, 64, 64, beta_free=True, n_segments=4096)["n_segments"] == 4096
    bad_bv = api.gdr_options(0.0, 0, 48, None, 0, None)
    assert _fwd(lib, ok, opt=bad_bv) == -1
    bad_scale = api.gdr_options(float("nan"), 0, 0, None, 0, None)
    assert _fwd(lib, ok, opt=bad_scale) == -1
    assert _fwd(lib, api.make_dims(1, 128, 2, 64, 64, flags=4)) == -1   # unknown flag bit


def test_host_entry_checks_host_seqlens_before_any_gpu_work(lib):
    """gdr_chunk_fwd_host reads cu_seqlens on the host: a table that does not
    rise from 0 to T is rejected with GDR_ERR_SEQLENS before any copy."""
    p = lambda x: ctypes.c_void_p(0x1000 * x)
    dims = api.make_dims(1, 128, 2, 64, 64, N=3)
    for table in ([0, 64, 32, 128], [1, 64, 96, 128], [0, 64, 96, 127]):
        cu = (ctypes.c_int32 * 4)(*table)
        rc = lib.gdr_chunk_fwd_host(ctypes.byref(dims), p(1), p(1), p(1), p(1), None,
                                    ctypes.cast(cu, ctypes.c_void_p), None, p(1), None, 0, None)
        assert rc == -5, table
    d64 = api.make_dims(1, 128, 2, 64, 64, N=3, flags=api.GDR_SEQLENS_I64)
    cu = (ctypes.c_int64 * 4)(0, 96, 64, 128)
    rc = lib.gdr_chunk_fwd_host(ctypes.byref(d64), p(1), p(1), p(1), p(1), None,
                                ctypes.cast(cu, ctypes.c_void_p), None, p(1), None, 0, None)
    assert rc == -5


def _bwd(lib, dims, q=1, do=1, dq=1, dg=1, beta=None, dbeta=None, cu=None, opt=None,
         n_segments=0):
    p = lambda x: None if x is None else ctypes.c_void_p(0x1000 * x)
    return lib.gdr_chunk_bwd(ctypes.byref(dims), p(q), p(1), p(1), p(1), p(beta), p(cu), None,
                             p(do), None, p(dq), p(1), p(1), p(dg), p(dbeta), None, n_segments,
                             None if opt is None else ctypes.byref(opt), None)


def test_backward_argument_checks_reject_before_any_gpu_work(lib):
    ok = api.make_dims(1, 128, 2, 64, 64)
    assert _bwd(lib, ok, q=None) == -1
    assert _bwd(lib, ok, do=None) == -1
    assert _bwd(lib, ok, dq=None) == -1
    assert _bwd(lib, ok, dg=None) == -1
    assert _bwd(lib, ok, beta=1, dbeta=None) == -1      # dbeta exactly when beta
    assert _bwd(lib, ok, beta=None, dbeta=1) == -1
    assert _bwd(lib, api.make_dims(1, 128, 2, 60, 64)) == -2
    assert _bwd(lib, api.make_dims(1, 128, 2, 64, 64, N=3)) == -1  # varlen needs cu
    # the tensor-core route takes BF16, K = V = 128, the delta rule; a route
    # number past 2 is invalid
    assert _bwd(lib, ok, opt=api.gdr_options(0.0, 2, 0, None, 0, None)) == -2
    assert _bwd(lib, ok, opt=api.gdr_options(0.0, 3, 0, None, 0, None)) == -1
    assert _bwd(lib, ok, opt=api.gdr_options(float("nan"), 0, 0, None, 0, None)) == -1
    assert _bwd(lib, ok, n_segments=-1) == -1
    assert _bwd(lib, ok, n_segments=1000) == -2
    assert pkg.gdr_kernel_name(16) == "bwd_gram" and pkg.gdr_kernel_name(19) == "bwd_local"


def test_backward_workspace_size_grows_with_the_problem(lib):
    a = pkg.gdr_bwd_workspace_size(1, 1024, 4, 128, 128)
    b = pkg.gdr_bwd_workspace_size(1, 2048, 4, 128, 128)
    c = pkg.gdr_bwd_workspace_size(1, 1024, 4, 128, 128, beta_free=True)
    assert 0 < c < a < b
    assert pkg.gdr_bwd_workspace_size(1, 1024, 4, 60, 128) == 0
    # a split keeps per-segment summaries as well
    assert pkg.gdr_bwd_workspace_size(1, 1024, 4, 128, 128, n_segments=4) > a


def _rec(lib, dims, q=1, state=1, n_states=4, idx=None, cu=None):
    p = lambda x: None if x is None else ctypes.c_void_p(0x1000 * x)
    return lib.gdr_recurrent_fwd(ctypes.byref(dims), p(q), p(1), p(1), p(1), None, p(cu),
                                 p(state), ctypes.c_int64(n_states), p(idx), p(1), None, None)


def test_recurrent_argument_checks_reject_before_any_gpu_work(lib):
    ok = api.make_dims(4, 1, 2, 64, 64)
    assert _rec(lib, ok, q=None) == -1
    assert _rec(lib, ok, state=None) == -1
    assert _rec(lib, ok, n_states=0) == -1
    assert _rec(lib, ok, n_states=3) == -1        # row n for 4 sequences needs 4 rows
    assert _rec(lib, api.make_dims(4, 1, 2, 60, 64)) == -2
    assert _rec(lib, api.make_dims(1, 8, 2, 64, 64, N=3)) == -1  # varlen needs cu_seqlens
    assert pkg.gdr_error_string(-7) == "state index out of range"


def test_plan_query_is_deterministic_and_valid():
    for dims in [(1, 256, 2, 64, 64, 0, 0), (1, 10456, 16, 128, 128, 32, 1),
                 (1, 16384, 16, 128, 128, 0, 1), (1, 65536, 1, 128, 128, 0, 1),
                 (2, 8192, 4, 256, 512, 0, 1)]:
        a = pkg.gdr_plan_query(*dims)
        b = pkg.gdr_plan_query(*dims)
        assert a == b
        B, T, H, K, V = dims[:5]
        assert V % a["bv"] == 0
        assert a["path"] == 2 or K % a["bv"] == 0
        assert 1 <= a["n_segments"] <= 64
    # an explicit segment count is taken as given
    assert pkg.gdr_plan_query(1, 16384, 16, 128, 128, n_segments=4)["n_segments"] == 4
    # a long single sequence with few heads is split; a wide batch is not
    assert pkg.gdr_plan_query(1, 65536, 1, 128, 128)["n_segments"] > 1
    assert pkg.gdr_plan_query(1, 10456, 16, 128, 128, N=32)["n_segments"] == 1
    # the tensor-core plan's cost model picks the counts measured fastest on
    # GB300 for the four split workloads (segments that fill the 152 SMs)
    best = {(1, 16384, 16, 128, 128, False): 9, (1, 65536, 8, 128, 128, False): 19,
            (1, 65536, 1, 128, 128, False): 54, (2, 8192, 4, 256, 512, True): 4}
    for (B, T, H, K, V, bf), s in best.items():
        assert pkg.gdr_plan_query(B, T, H, K, V, beta_free=bf)["n_segments"] == s
    # and for the two skewed batches (one 16K-token sequence among short
    # ones, the max_len hint given) at the common segment length: 9 of
    # 6 / 8 / 9 / 12 / 16 at 16 heads, 16 of 12 / 16 / 24 / 32 at 4 heads
    assert pkg.gdr_plan_query(1, 50360, 16, 128, 128, N=101, max_len=16384)["n_segments"] == 9
    assert pkg.gdr_plan_query(1, 26421, 4, 128, 128, N=32, max_len=16384)["n_segments"] == 16


def test_plan_reports_the_composition():
    """The segment split's ordered composition as the plan reports it (the
    cost model of GB300 timings, 152 SMs): the tensor cores' single pass for
    the 64K x 8-head and 16K x 16-head splits, their two-level form in groups
    of 7 for one 64K-token head at 54 segments, the CUDA-core pass for one
    head at 4 segments; none without a split, on the CUDA-core path, or in
    the beta-free mode (its composition is element-wise)."""
    q = pkg.gdr_plan_query
    assert q(1, 65536, 8, 128, 128)["compose"] == 1
    assert q(1, 65536, 1, 128, 128)["compose"] == 7
    assert q(1, 16384, 16, 128, 128)["compose"] == 1
    assert q(1, 16384, 1, 128, 128, n_segments=4)["compose"] == 0
    assert q(1, 10456, 16, 128, 128, N=32)["compose"] == 0
    assert q(2, 8192, 4, 256, 512, beta_free=True)["compose"] == 0
    assert q(1, 4096, 2, 64, 64, dtype=0, n_segments=4)["compose"] == 0


def test_plan_keys_on_the_longest_sequence():
    """Varlen plans read the longest sequence from the max_len hint
    (cu_seqlens is device data): at 4 heads one 16K-token sequence among 31
    short ones is split, the same batch without the hint (mean length 822)
    or a uniform batch is not, and a negative hint is rejected."""
    skew = (1, 26304, 4, 128, 128)  # one 16K-token sequence and 31 of 320 tokens
    assert pkg.gdr_plan_query(*skew, N=32)["n_segments"] == 1
    assert pkg.gdr_plan_query(*skew, N=32, max_len=16384)["n_segments"] > 1
    # with 16 heads and 100 short sequences too: one segment length for all
    # sequences leaves the short ones whole, so only the long one's 16 heads
    # are pre-scanned and composed
    skew16 = pkg.gdr_plan_query(1, 50360, 16, 128, 128, N=101, max_len=16384)
    assert skew16["n_segments"] > 1 and skew16["compose"] == 1
    # the beta-free mode alike (K = 256, V = 512, 4 heads): its composition
    # walks the long sequence's states only
    gla = (1, 26005, 4, 256, 512)
    assert pkg.gdr_plan_query(*gla, N=32, beta_free=True, max_len=16384)["n_segments"] > 1
    assert pkg.gdr_plan_query(*gla, N=32, beta_free=True)["n_segments"] == 1
    assert pkg.gdr_plan_query(1, 10456, 16, 128, 128, N=32, max_len=512)["n_segments"] == 1
    # a hint longer than the batch is clamped to it: one sequence of T tokens
    assert (pkg.gdr_plan_query(1, 16384, 16, 128, 128, N=1, max_len=1 << 40)
            == pkg.gdr_plan_query(1, 16384, 16, 128, 128))
    # the CUDA-core rule (FP32 inputs, fewer than two chains an SM) splits on
    # the longest sequence too
    one_head = (1, 26304, 1, 128, 128)
    assert pkg.gdr_plan_query(*one_head, N=32, dtype=0, max_len=16384)["n_segments"] > 1
    assert pkg.gdr_plan_query(*one_head, N=32, dtype=0)["n_segments"] == 1
    with pytest.raises(pkg.GdrError):
        pkg.gdr_plan_query(*skew, N=32, max_len=-1)


def test_cuda_core_plan_rules():
    """The CUDA-core plan (FP32 inputs): 32-column value tiles, 16 when the
    sequences are too short to split and 32-column tiles leave SMs without a
    chain; up to 64 segments for a long sequence with few heads (the
    measurements behind each rule are stated beside pick_bv and
    auto_segments)."""
    q = lambda *a, **k: pkg.gdr_plan_query(*a, dtype=0, **k)
    assert q(1, 256, 2, 64, 64) == {"path": 1, "bv": 16, "n_segments": 1, "compose": 0}
    assert q(1, 10456, 16, 128, 128, N=32) == {"path": 1, "bv": 32, "n_segments": 1, "compose": 0}
    assert q(1, 16384, 16, 128, 128) == {"path": 1, "bv": 32, "n_segments": 8, "compose": 0}
    assert q(1, 65536, 1, 128, 128) == {"path": 1, "bv": 32, "n_segments": 64, "compose": 0}
    assert q(2, 8192, 4, 256, 512, beta_free=True) == {"path": 1, "bv": 32, "n_segments": 4, "compose": 0}


def test_fp16_inputs_plan_the_cuda_core_path():
    """FP16 (dtype 2) goes to path 1 by default (FP32 arithmetic); the
    tensor-core kernels take it only when forced, on BF16 copies."""
    plan = pkg.gdr_plan_query(1, 1000, 16, 128, 128, N=4, dtype=api.GDR_F16)
    assert plan["path"] == 1
    assert pkg.gdr_workspace_size(1, 1000, 16, 128, 128, N=4, dtype=api.GDR_F16) > 0


def test_workspace_size_scales_with_problem():
    # CUDA-core path keeps W, U, h_pre, v_new in HBM: grows with tokens
    small = pkg.gdr_workspace_size(1, 256, 2, 64, 64, dtype=0)
    big = pkg.gdr_workspace_size(1, 16384, 16, 64, 64, dtype=0, n_segments=1)
    assert 0 < small < big
    # tensor-core path: one 74,752-byte record (the scan's stage image) per
    # (chunk, head) plus the chunk table, and the FP32 segment summaries when
    # the sequence is split
    tc = pkg.gdr_workspace_size(1, 16384, 16, 128, 128, n_segments=1)
    tc_seg = pkg.gdr_workspace_size(1, 16384, 16, 128, 128, n_segments=16)
    records = 256 * 16 * 74752
    assert records < tc < records + 64 * 1024
    assert tc_seg >= tc + 16 * 16 * 3 * 128 * 128 * 4
    gla = pkg.gdr_workspace_size(1, 16384, 16, 128, 128, beta_free=True, n_segments=1)
    assert gla > 0
    assert pkg.gdr_workspace_size(1, 256, 2, 60, 64) == 0  # unsupported -> 0


def test_binding_rejects_misuse_before_calling_the_library(lib):
    """The Python binding checks devices, dtypes and shapes before any CUDA
    call: host tensors to the device entry points, mixed input dtypes, a
    do of the wrong shape."""
    import torch
    q = torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16)
    g = torch.zeros(1, 64, 2)
    with pytest.raises(ValueError):
        pkg.gdr_chunk_fwd(q, q, q, g)
    with pytest.raises(ValueError):
        pkg.gdr_chunk_bwd(q, q, q, g, None, q)
    with pytest.raises(ValueError):
        pkg.chunk_gated_delta_rule(q, q, q, g)
    with pytest.raises(TypeError):  # k in another dtype than q
        pkg.gdr_chunk_fwd_host(q, q.float(), q, g)
    with pytest.raises(TypeError):  # g must be float32
        pkg.gdr_chunk_fwd_host(q, q, q, g.double())
    with pytest.raises(ValueError):  # host entry wants host tensors; meta is not one
        pkg.gdr_chunk_fwd_host(q.to("meta"), q, q, g)


def test_stride_validation():
    """Tensor strides in gdr_dims: a pair is both zero or both positive; o's
    rows may not overlap; the host entry takes contiguous tensors only.
    Checked on the host before any CUDA call."""
    lib = pkg.load_library()
    p = ctypes.c_void_p(0x1000)

    def fwd(dims):
        return lib.gdr_chunk_fwd(ctypes.byref(dims), p, p, p, p, p, None, None, p, p, 0, None)

    d = api.make_dims(1, 128, 2, 64, 64)
    d.q_stride[:] = (0, 64)
    assert fwd(d) == -1                      # half a pair
    d = api.make_dims(1, 128, 2, 64, 64)
    d.o_stride[:] = (64, 32)                 # heads 32 apart: rows of 64 overlap
    assert fwd(d) == -1
    d = api.make_dims(1, 128, 2, 64, 64)
    d.o_stride[:] = (64, 64)                 # two heads on one row
    assert fwd(d) == -1
    d = api.make_dims(1, 128, 2, 64, 64)
    d.k_stride[:] = (-384, 64)
    assert fwd(d) == -1
    # a fused [B, T, 3, H, K] projection's views are fine; the host entry
    # refuses them (it copies whole contiguous buffers)
    d = api.make_dims(1, 128, 2, 64, 64)
    for f in ("q_stride", "k_stride", "v_stride"):
        getattr(d, f)[:] = (3 * 2 * 64, 64)
    assert pkg.gdr_plan_query(1, 128, 2, 64, 64)["path"] in (1, 2)
    assert lib.gdr_chunk_fwd_host(ctypes.byref(d), p, p, p, p, p, None, None, p, p, 0,
                                  None) == -2
    # head-major o (tokens inside heads) is a valid layout
    d = api.make_dims(1, 128, 2, 64, 64)
    d.o_stride[:] = (64, 128 * 64)
    assert api.gdr_dims.o_stride.size == 16 and d.o_stride[1] == 8192
