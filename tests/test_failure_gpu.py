"""Failure detection on the GPU without a fault: a kernel wait that runs out is reported through
the device error word and leaves the device usable.

fa_selftest_wait_timeout makes one warp wait, with the same bounded wait the attention kernels
use, on a barrier that nothing completes; the wait gives up after the given limit and records
the timeout. No trap, no fault, no hang: the limit here is 20 ms.
"""
import numpy as np
import pytest

import oracle
from gpu_util import o_bound, to_device
from io_aware_attention_fa2_gb300.inputs import make_qkv, softmax_scale

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = -8


def test_wait_that_runs_out_is_reported_and_cleared():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = binding.load_library()
    stream = torch.cuda.current_stream()
    assert binding.device_error() == 0                      # nothing pending before
    assert lib.fa_selftest_wait_timeout(20000, stream.cuda_stream) == 0
    assert binding.device_error() == FA_ERR_TIMEOUT         # reported ...
    assert binding.device_error() == 0                      # ... and cleared by the read


def test_device_usable_after_a_timeout():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    lib = binding.load_library()
    assert lib.fa_selftest_wait_timeout(5000, torch.cuda.current_stream().cuda_stream) == 0
    assert binding.device_error() == FA_ERR_TIMEOUT
    B, H, N, d = 1, 2, 257, 64
    qb, kb, vb = make_qkv(B, H, N, d, "bf16", seed=77)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    binding.fa_fwd(q, k, v, o, lse, True, softmax_scale(d))
    assert binding.device_error() == 0
    o_ref, _ = oracle.attention(qb, kb, vb, True, softmax_scale(d), dtype="bf16")
    assert (np.abs(o.double().cpu().numpy() - o_ref) - o_bound(o_ref, "bf16")).max() <= 0
