"""FP16 inputs (GDR_F16): the plan routes them to the CUDA-core path (FP32
arithmetic; the tensor-core kernels take BF16) and to the per-token
recurrence.  Parity against the FP64 oracle on the same FP16-rounded
inputs: o is rounded to FP16 once (rel-L2 <= 2e-3), ht is FP32 arithmetic
(<= 1e-5).  All calls go through the C ABI."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import TOL_F32, assert_parity, rel_l2_masked, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS
TOL_O_F16 = 2e-3
LENS = [1, 63, 64, 65, 130, 7, 0, 200]


def check(x, **kw):
    o, ht = run_gpu(x, **kw)
    ro, rht = run_oracle(x)
    assert o.dtype == torch.float16
    assert_parity(x, o, ht, ro, rht, TOL_O_F16, TOL_F32, label=f"fp16 {kw}")


@pytest.mark.parametrize("S", [1, 4])
def test_varlen_delta(S):
    w = synthetic.small(W["wide_varlen_bf16"], H=2, dtype="f16", with_h0=True)
    check(synthetic.make_inputs(w, lengths=LENS), n_segments=S)


@pytest.mark.parametrize("S", [1, 2])
def test_beta_free(S):
    w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=2, dtype="f16", T=300)
    check(synthetic.make_inputs(w), n_segments=S)


def test_recurrent_fp16():
    w = synthetic.small(W["decode_bf16"], H=2, dtype="f16")
    x = synthetic.make_inputs(w, lengths=[1, 3, 0, 2])
    pool, idx = synthetic.make_state_pool(x, 7)
    d = to_dev(x)
    p = pool.cuda()
    o = pkg.gdr_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                              cu_seqlens=d["cu_seqlens"], state=p, state_indices=idx.cuda())
    torch.cuda.synchronize()
    ro, rht = run_oracle(x)
    assert_parity(x, o, p.cpu()[idx.long()], ro, rht, TOL_O_F16, TOL_F32, label="fp16 recurrent")


TOL_BF16_OPERANDS = 6e-3  # the BF16 bar: the tensor-core kernels take BF16 operands


@pytest.mark.parametrize("case", ["delta_varlen", "beta_free"])
def test_tensor_core_path_on_fp16_inputs(case):
    """force_path=2 with FP16 inputs: the kernels read BF16 copies of q, k, v
    and o comes back in FP16.  Against the oracle on the FP16 inputs the
    result meets the BF16 bar (BF16 operands); against the BF16 path run on
    the same BF16-rounded inputs it is bit-identical (ht) and equal after
    o's final conversion to FP16."""
    if case == "delta_varlen":
        w = synthetic.small(W["wide_varlen_bf16"], H=2, dtype="f16", with_h0=True)
        x = synthetic.make_inputs(w, lengths=LENS)
    else:
        w = synthetic.small(W["gla_k256_v512_bf16"], K=128, V=256, H=2, dtype="f16", T=300)
        x = synthetic.make_inputs(w)
    o, ht = run_gpu(x, force_path=2)
    assert o.dtype == torch.float16
    o2, ht2 = run_gpu(x, force_path=2, n_segments=2)  # the split on the same copies
    ro, rht = run_oracle(x)
    assert_parity(x, o2, ht2, ro, rht, TOL_BF16_OPERANDS, label=f"{case} split")
    assert_parity(x, o, ht, ro, rht, TOL_BF16_OPERANDS, label=case)
    xb = dict(x)
    for name in ("q", "k", "v"):
        xb[name] = x[name].to(torch.bfloat16)
    ob, htb = run_gpu(xb, force_path=2)
    assert torch.equal(ht, htb)
    assert torch.equal(o, ob.to(torch.float16))
