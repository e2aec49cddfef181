"""Standard (materialised) attention on the GPU, the comparison the pages make against the
fused kernel ("FlashAttention V2 核心原理与架构设计" §3.1: S = QK^T and P = softmax(S) written
to and read back from HBM). The benchmark's ``time_standard_attention`` (fp32 scores and
softmax, P rounded to the input type for P V: the fused kernel's precision) must compute the
same attention as the oracle under the same bar as the fused kernel, element by element;
otherwise its timings would compare the kernel with a wrong baseline.
"""
import pytest

import oracle
from gpu_util import assert_close, attention_aux, to_device
from io_aware_attention_fa2_gb300.inputs import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["n1k_d128", "n1k_d64_causal"])
def test_standard_attention_matches_oracle(name):
    import torch

    import bench
    w = WORKLOADS[name]
    qb, kb, vb = make_workload(w)
    q, k, v = (to_device(x, w.dtype) for x in (qb, kb, vb))
    flush = torch.empty(1 << 20, dtype=torch.uint8, device=q.device)
    ms, o_std, how = bench.time_standard_attention(q, k, v, w, 3, flush,
                                                   torch.cuda.current_stream())
    assert ms > 0 and o_std.shape == q.shape and o_std.dtype == q.dtype and "fp32" in how
    o_ref, lse_ref = oracle.attention(qb, kb, vb, w.causal, w.scale, dtype=w.dtype)
    a_ref, _ = attention_aux(qb, kb, vb, w.causal, w.scale, w.dtype)
    # the standard arm has no LSE: its O alone against the bar
    assert_close(o_std.double().cpu().numpy(), lse_ref, o_ref, lse_ref, "standard " + name,
                 w.dtype, a_ref)

