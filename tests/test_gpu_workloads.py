"""GPU parity at the full workload sizes, in the plan the benchmark times
(n_segments=0) and at forced segment counts.  Where the FP64 oracle over
every (sequence, head) pair would take too long, a fixed sample of pairs is
checked element by element (the oracle computes pairs independently)."""
import numpy as np
import pytest

from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import TOL_BF16, assert_parity, run_gpu, run_oracle, sample_mask

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS

_cache = {}


def reference(name, pairs=None):
    key = (name, tuple(pairs) if pairs else None)
    if key not in _cache:
        x = synthetic.make_inputs(W[name])
        mask = None if pairs is None else sample_mask(x["N"], x["H"], pairs)
        _cache[key] = (x, run_oracle(x, pair_mask=mask))
    return _cache[key]


def check(name, pairs=None, **kw):
    x, (ro, rht) = reference(name, pairs)
    o, ht = run_gpu(x, **kw)
    assert_parity(x, o, ht, ro, rht, TOL_BF16, label=f"{name} {kw}")


def test_wide_varlen_all_pairs():
    check("wide_varlen_bf16", n_segments=0)


@pytest.mark.parametrize("S", [0, 1, 2, 4, 8, 16])
def test_long_16k(S):
    check("long_16k_bf16", pairs=[(0, 0), (0, 5), (0, 10), (0, 15)], n_segments=S)


@pytest.mark.parametrize("S", [0, 1, 16])
def test_stress_64k_h8(S):
    check("stress_64k_h8_bf16", pairs=[(0, 0), (0, 7)], n_segments=S)


@pytest.mark.parametrize("S", [0, 1, 16])
def test_stress_64k_h1(S):
    check("stress_64k_h1_bf16", n_segments=S)


@pytest.mark.parametrize("S", [0, 1, 8, 128])
def test_gla_k256_v512(S):
    check("gla_k256_v512_bf16", pairs=[(0, 0), (1, 3)], n_segments=S)


@pytest.mark.parametrize("S", [0, 1])
def test_skewed_varlen(S):
    """One 16K-token sequence (number 50) among 100 of 128..512 tokens: with
    the longest-sequence hint the plan splits (S = 0), the serial scan is
    the reference plan; pairs on the long sequence and on short ones."""
    check("skewed_varlen_bf16", pairs=[(50, 0), (50, 15), (0, 3), (100, 7)], n_segments=S)


@pytest.mark.parametrize("S", [0, 1])
def test_skewed_varlen_h4(S):
    """One 16K-token sequence (number 16) among 31 short ones at 4 heads: the
    longest-sequence hint makes the plan split (S = 0)."""
    check("skewed_varlen_h4_bf16", pairs=[(16, 0), (16, 3), (0, 1), (31, 2)], n_segments=S)


@pytest.mark.parametrize("S", [0, 1])
def test_skewed_gla_h4(S):
    """The beta-free mode (K = 256, V = 512, h0 in) on one 16K-token sequence
    (number 16) among 31 short ones: the plan splits the long sequence alone
    at the common segment length (S = 0); pairs on the long sequence and on
    short ones."""
    check("skewed_gla_h4_bf16", pairs=[(16, 0), (16, 3), (0, 1), (31, 2)], n_segments=S)
