"""FP16 inputs (GDR_F16): the plan routes them to the CUDA-core path (FP32
arithmetic; the tensor-core kernels take BF16) and to the per-token
recurrence.  Parity against the FP64 oracle on the same FP16-rounded
inputs: o is rounded to FP16 once (rel-L2 <= 2e-3), ht is FP32 arithmetic
(<= 1e-5).  All calls go through the C ABI."""
import pytest
import torch

import chunked_gated_delta_rule_gb300 as pkg
from chunked_gated_delta_rule_gb300 import synthetic
from gpu_util import TOL_F32, rel_l2_masked, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

W = synthetic.WORKLOADS
TOL_O_F16 = 2e-3
LENS = [1, 63, 64, 65, 130, 7, 0, 200]


def check(x, **kw):
    o, ht = run_gpu(x, **kw)
    ro, rht = run_oracle(x)
    assert o.dtype == torch.float16
    eo, eh = rel_l2_masked(o, ro), rel_l2_masked(ht, rht)
    assert eo <= TOL_O_F16 and eh <= TOL_F32, (eo, eh)


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
    assert rel_l2_masked(o, ro) <= TOL_O_F16
    assert rel_l2_masked(p.cpu()[idx.long()], rht) <= TOL_F32
