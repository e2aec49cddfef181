"""Full-tensor parity of the long workloads with the fp64 oracle: every element of O and LSE.

The three long configurations (B=2 H=16 N=8192 d=128 bf16 causal; B=1 H=8 N=32768 d=128 bf16
causal; B=16 H=32 N=2000 d=128 fp16 with Q x8 and 1 % of K rows x10, non-causal), each in one
fa_fwd call exactly as the benchmark launches it, compared element by element with the oracle's
unrounded fp64 result under the one bar of ``oracle.tolerance`` (tiling does not change the
result: "FlashAttention 优化原理与实现要点解析" §1 and §4.3). The oracle is the plain
row-by-row definition, so each case costs tens of seconds of host time.
"""
import numpy as np
import pytest

import oracle
from gpu_util import to_device
from io_aware_attention_fa2_gb300.inputs import WORKLOADS, make_workload
from oracle.tolerance import stats

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["n8k_d128_causal", "n32k_d128_causal",
                                  "n2000_d128_fp16_stress"])
def test_workload_every_element(name):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    q, k, v = (to_device(x, w.dtype) for x in (qb, kb, vb))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, w.causal, w.scale)
    assert binding.device_error() == 0
    o_gpu = o.cpu().float().double().numpy()
    lse_gpu = lse.cpu().double().numpy()
    del q, k, v, o, lse
    o_ref, lse_ref = oracle.attention(qb, kb, vb, w.causal, w.scale, dtype=w.dtype)
    st = stats(o_gpu, lse_gpu, o_ref, lse_ref, w.dtype)
    print(name, st)
    assert st["ok"], (name, st)
