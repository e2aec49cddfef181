"""Parity of the split-K/V forward (fa_fwd_splitkv) with the fp64 oracle: fewer queries than
keys (decoding shapes), K/V ranges cut into several parts and merged, masks, and parts that
hold no key at all."""
import numpy as np
import pytest

import oracle
from gpu_util import MAX_ABS_LSE, MAX_ABS_O, REL_L2_O, o_bound, to_device
from io_aware_attention_fa2_gb300.inputs import make_qkv, softmax_scale

pytestmark = pytest.mark.gpu


def run_split(qb, kb, vb, dtype, causal, splits, window=(-1, -1), lens=None):
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
    B, Nq, H, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=q.device)
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=q.device)
    binding.fa_fwd_splitkv(q, k, v, o, lse, causal, softmax_scale(d), splits, None, None,
                           window, lens_t)
    assert binding.device_error() == 0
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(o, lse, o_ref, lse_ref, what, dtype):
    assert np.isfinite(o).all(), what
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    d_o = o - o_ref
    assert (np.abs(d_o) - o_bound(o_ref, dtype)).max() <= 0, (what, float(np.abs(d_o).max()))
    if np.linalg.norm(o_ref) > 0:
        assert np.linalg.norm(d_o) / np.linalg.norm(o_ref) <= REL_L2_O, what
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= MAX_ABS_LSE, what


def case(B, H, Nq, Nk, d, dtype, causal, splits, seed, window=(-1, -1), lens=None):
    qb, kb, vb = make_qkv(B, H, Nq, d, dtype, seed, Nk=Nk)
    o, lse = run_split(qb, kb, vb, dtype, causal, splits, window, lens)
    o_ref, lse_ref = oracle.attention(qb, kb, vb, causal, softmax_scale(d), dtype=dtype,
                                      window=window, seqlens_k=lens)
    check(o, lse, o_ref, lse_ref, (B, H, Nq, Nk, d, dtype, causal, splits, window, lens), dtype)


@pytest.mark.parametrize("Nk", [1, 127, 1000, 4173])
@pytest.mark.parametrize("splits", [1, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_decode(Nk, splits, causal):
    case(2, 4, 1, Nk, 128, "bf16", causal, splits, seed=600 + Nk)


@pytest.mark.parametrize("Nk", [1, 1000])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_d64(Nk, splits, causal):
    """One query at d = 64: unsplit it takes the one-Q-tile kernel, split the two-tile one."""
    case(2, 4, 1, Nk, 64, "bf16", causal, splits, seed=650 + Nk)


@pytest.mark.parametrize("Nq,Nk", [(16, 2000), (129, 700), (300, 300), (513, 1100)])
@pytest.mark.parametrize("splits", [1, 4])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_fewer_queries(Nq, Nk, splits, causal, d):
    case(2, 2, Nq, Nk, d, "bf16", causal, splits, seed=700 + Nq + Nk)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_split_masks(dtype):
    case(3, 2, 40, 1500, 128, dtype, True, 5, seed=800, window=(600, -1), lens=[1500, 900, 10])
    case(2, 2, 700, 700, 64, dtype, False, 3, seed=801, window=(100, 50), lens=[650, 700])


def test_more_parts_than_tiles():
    """16 parts over 3 K/V tiles: most parts are empty (LSE -inf) and the merge skips them."""
    case(1, 2, 5, 300, 128, "bf16", False, 16, seed=802)
    case(2, 1, 1, 129, 64, "bf16", True, 128, seed=803)


def test_split_matches_unsplit_square():
    """For Nq = Nk, splitting the K/V range changes only rounding."""
    import torch

    from io_aware_attention_fa2_gb300 import binding
    qb, kb, vb = make_qkv(2, 3, 900, 128, "bf16", seed=804)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(2, 3, 900, device="cuda")
    l2 = torch.empty_like(l1)
    binding.fa_fwd(q, k, v, o1, l1, True, softmax_scale(128))
    binding.fa_fwd_splitkv(q, k, v, o2, l2, True, softmax_scale(128), 4)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * MAX_ABS_O
    assert (l1 - l2).abs().max().item() <= MAX_ABS_LSE


def test_long_decode_full():
    """One decoding step against 32768 keys, every head, with the library's part count."""
    import torch

    from io_aware_attention_fa2_gb300 import attention_forward
    qb, kb, vb = make_qkv(4, 8, 1, 128, "bf16", seed=805, Nk=32768)
    q, k, v = (to_device(x, "bf16") for x in (qb, kb, vb))
    o, lse = attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(qb, kb, vb, True, softmax_scale(128), dtype="bf16")
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, "decode 32K",
          "bf16")


def test_workspace_too_small_on_gpu():
    import torch

    from io_aware_attention_fa2_gb300 import binding
    q = torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1024, 2, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 4, device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.FaError) as e:
        binding.fa_fwd_splitkv(q, k, k, o, lse, False, 0.088, 4, ws)
    assert e.value.code == -11
    torch.cuda.synchronize()
    assert float(o.float().abs().sum()) == 0.0
