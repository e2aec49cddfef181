"""The seeded input generator (CPU only): determinism, rounding, the stress recipe."""
import numpy as np
import torch

from io_aware_attention_fa2_gb300.inputs import (WORKLOADS, make_qkv, round_to_bits,
                                                 sample_rows, softmax_scale)


def test_deterministic_and_seed_sensitive():
    a = make_qkv(1, 2, 33, 64, "bf16", seed=5)
    b = make_qkv(1, 2, 33, 64, "bf16", seed=5)
    c = make_qkv(1, 2, 33, 64, "bf16", seed=6)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[0], c[0])
    assert a[0].shape == (1, 33, 2, 64) and a[0].dtype == np.uint16


def test_rounding_is_nearest_even():
    x = np.random.Generator(np.random.PCG64(0)).standard_normal(100000) * 37.0
    # bf16: float64 -> float32 (nearest-even), then float32 -> bf16 nearest-even, as torch does
    bits = round_to_bits(x, "bf16")
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(bits.view(np.int16), want)
    # fp16: one rounding from float64; no representable neighbour is closer, ties go to even
    h = round_to_bits(x, "fp16").view(np.float16)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h, np.float16(-np.inf)).astype(np.float64)
    err = np.abs(x - h.astype(np.float64))
    assert (err <= np.abs(x - up)).all() and (err <= np.abs(x - dn)).all()
    tie = (err == np.abs(x - up)) | (err == np.abs(x - dn))
    assert (h[tie].view(np.uint16) & 1 == 0).all()


def test_stress_recipe_scales_k_rows():
    B, H, N, d = 2, 3, 200, 64
    plain = make_qkv(B, H, N, d, "fp16", seed=9)
    stress = make_qkv(B, H, N, d, "fp16", seed=9, q_scale=8.0, k_outlier_frac=0.01,
                      k_outlier_scale=10.0)
    q0 = plain[0].view(np.float16).astype(np.float64)
    q1 = stress[0].view(np.float16).astype(np.float64)
    assert np.allclose(q1, 8 * q0, rtol=2e-3, atol=1e-6)
    k0 = plain[1].view(np.float16).astype(np.float64)
    k1 = stress[1].view(np.float16).astype(np.float64)
    ratio = np.abs(k1).sum(-1) / np.abs(k0).sum(-1)      # [B, N, H]
    scaled = ratio > 5
    assert (scaled.sum(axis=1) == 2).all()               # round(0.01 * 200) rows per (b, h)
    assert np.array_equal(stress[2], plain[2])


def test_named_workloads():
    assert WORKLOADS["n8k_d128_causal"].causal and WORKLOADS["n8k_d128_causal"].N == 8192
    assert softmax_scale(128) == float(np.float32(1 / np.sqrt(128)))
    rows = sample_rows(2, 3, 300, 5, seed=1)
    assert rows.shape[1] == 3 and rows[:, 2].max() < 300
    assert {(0, 0, 0), (1, 2, 299)} <= {tuple(r) for r in rows}
