"""The tensor-core building blocks on the GPU, compared with PyTorch: every
tcgen05 operand layout the fused path issues (K-major / MN-major, 128-byte
swizzle, M=128, N=64/128, K=64/128) and the TMA box load with its swizzle
address map (including rows past the end, which read as zero)."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import api

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,Kd", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1)])
def test_umma_layouts(N, Kd, a_mn, b_mn):
    pkg.load_library()
    g = torch.Generator(device="cuda").manual_seed(N * 7 + Kd + 3 * a_mn + b_mn)
    A = torch.randn(128, Kd, generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, Kd, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = api.gdr_selftest_umma(A, B, a_mn, b_mn, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.double() @ B.double().T
    err = ((D.double() - ref).norm() / ref.norm()).item()
    assert err < 1e-5, err


@pytest.mark.parametrize("t0,h,k0", [(0, 0, 0), (5, 2, 64), (100, 1, 8), (130, 3, 64)])
def test_tma_swizzled_box(t0, h, k0):
    pkg.load_library()
    T, H, K = 150, 4, 128
    src = torch.randn(T, H, K, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gdr_selftest_tma(src, t0, h, k0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    rows = min(64, T - t0)
    want[:rows] = src[t0:t0 + rows, h, k0:k0 + 64]
    assert torch.equal(out, want)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_blocked_triangular_inverse(seed):
    """The chain kernel's (I + A)^-1 (FP32 diagonal blocks, 3xTF32 warp MMAs
    off the diagonal) against a float64 library inverse, on A shaped like the
    chunk Gram matrix: beta_i e^{G_i - G_j} (k_i . k_j) with unit keys."""
    pkg.load_library()
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(64, 128, generator=g, dtype=torch.float64)
    k = k / k.norm(dim=1, keepdim=True)
    beta = torch.sigmoid(torch.randn(64, generator=g, dtype=torch.float64))
    G = torch.cumsum(torch.nn.functional.logsigmoid(torch.randn(64, generator=g,
                                                                dtype=torch.float64) + 3), 0)
    A = torch.tril(beta[:, None] * torch.exp(G[:, None] - G[None, :]) * (k @ k.T), -1)
    T = api.gdr_selftest_inverse(A.float().cuda())
    torch.cuda.synchronize()
    ref = torch.linalg.inv(torch.eye(64, dtype=torch.float64) + A.float().double())
    err = ((T.double().cpu() - ref).norm() / ref.norm()).item()
    assert err < 2e-6, err


def test_bounded_wait_times_out_cleanly():
    """A wait on a barrier nothing completes gives up after its limit,
    reports GDR_ERR_TIMEOUT and leaves the context usable."""
    pkg.load_library()
    status, done = api.gdr_selftest_timeout(1_000_000)
    assert status == -4 and done == 2
    # the context still works afterwards
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0
