"""The benchmark's FLOP counts on the CPU: the exact count of mask-allowed (query, key) pairs
against brute force on small shapes, and the unmasked formulas."""
import dataclasses
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from io_aware_attention_fa2_gb300.inputs import WORKLOADS, Workload  # noqa: E402


def brute_pairs(w):
    nq, nk = w.N, w.n_keys
    total = 0
    for b in range(w.B):
        length = w.seqlens_k[b] if w.seqlens_k else nk
        for i in range(nq):
            p = i + nk - nq
            for j in range(nk):
                ok = j < length and (not w.causal or j <= p)
                ok = ok and (w.window[0] < 0 or p - w.window[0] <= j)
                ok = ok and (w.window[1] < 0 or j <= p + w.window[1])
                total += ok
    return total * w.H


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window,lens", [((-1, -1), ()), ((5, -1), ()), ((3, 7), ()),
                                         ((-1, -1), (40, 9)), ((6, 2), (40, 0)),
                                         ((0, 0), (13, 40))])
def test_allowed_pairs_match_brute_force(causal, window, lens):
    w = Workload("t", 2, 3, 40, 64, "bf16", causal, 1, window=window, seqlens_k=lens)
    assert bench.allowed_pairs(w) == brute_pairs(w)
    if w.masked:
        assert bench.metric_flops(w) == 4.0 * 64 * brute_pairs(w)


def test_fewer_queries_than_keys():
    w = Workload("t", 2, 3, 7, 64, "bf16", True, 1, Nk=50)
    assert bench.allowed_pairs(w) == brute_pairs(w)
    assert bench.metric_flops(w) == 4.0 * 64 * brute_pairs(w)


def test_unmasked_headline_formula():
    w = WORKLOADS["n8k_d128_causal"]
    assert not w.masked
    assert bench.metric_flops(w) == 4.0 * 2 * 16 * 8192 * 8192 * 128 / 2


def test_masked_workloads_are_masked():
    for name in ("n8k_d128_window1k", "n8k_d128_padded"):
        w = WORKLOADS[name]
        assert w.masked and bench.metric_flops(w) < 4.0 * w.B * w.H * w.N * w.N * w.d
    w = dataclasses.replace(WORKLOADS["n8k_d128_padded"], B=2, N=64, seqlens_k=(64, 10))
    assert bench.allowed_pairs(w) == w.H * 64 * (64 + 10)


def test_reference_arm_reports_the_gpu_arms_metric():
    """Both arms of the bench print the same metric string for the same workload, so that their
    lines can be paired; the headline workload carries its own label."""
    import inspect
    src = inspect.getsource(bench.run_reference) + inspect.getsource(bench.run_gpu)
    assert src.count("metric_name(") == 2
    names = {bench.metric_name(w, False) for w in WORKLOADS.values()}
    assert bench.metric_name(WORKLOADS[bench.DEFAULT_WORKLOAD], False) in names
    assert len(names) == 2
    assert "bwd" in bench.metric_name(WORKLOADS[bench.DEFAULT_WORKLOAD], True)


def test_algorithmic_bytes_and_warm_l2_selection():
    """Q, K, V read and O written at 2 bytes an element plus the fp32 LSE, counted by hand for
    the headline shape; only the workloads whose data fits well inside L2 (the N = 256 and
    N = 1K ones) get the supplementary timing without the L2 flush."""
    w = WORKLOADS["n8k_d128_causal"]
    assert bench.algorithmic_bytes(w) == 4 * 2 * 8192 * 16 * 128 * 2 + 2 * 16 * 8192 * 4
    small = {n for n, x in WORKLOADS.items()
             if bench.algorithmic_bytes(x) < bench.WARM_L2_MAX_BYTES}
    assert small == {"tiny_n256_d64", "n1k_d64", "n1k_d64_causal", "n1k_d128"}
    assert bench.WARM_L2_MAX_BYTES < bench.L2_FLUSH_BYTES


def test_reference_arm_prints_the_gpu_arms_config(capsys):
    """The reference arm's JSON line carries exactly the config the GPU arm prints for the same
    workload (run here on the tiny workload with a bounded oracle sample)."""
    import json
    import types
    w = WORKLOADS["tiny_n256_d64"]
    args = types.SimpleNamespace(gpus=1, steps=3, warmup=3, ref_total_seconds=0.5)
    assert bench.run_reference(args, w) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.bench_config(w, 1)
    import inspect
    assert "bench_config(w, world)" in inspect.getsource(bench.run_gpu)
