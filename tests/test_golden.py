"""Stored fixtures under tests/golden/: numbers the pages print (cited in the fixture) and the
oracle's outputs on one tiny seeded input (a regression fixture written by
tests/golden/make_oracle_tiny.py, which calls only the oracle)."""
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
GOLDEN = os.path.join(HERE, "golden")


def _read_keys(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = line.split("=", 1)
                out[k.strip()] = v.strip()
    return out


def test_page_score_matrix_size():
    """One fp32 score matrix at N = 4096 is about 64 MB (64 MiB exactly)."""
    sys.path.insert(0, ROOT)
    import bench
    g = _read_keys("page_numbers.txt")
    n, e = int(g["score_matrix_n"]), int(g["score_matrix_elem_bytes"])
    assert bench.score_matrix_bytes(n, e) == int(g["score_matrix_about_mib"]) * 2 ** 20


def test_page_standard_attention_hbm_accesses():
    """The eight HBM accesses per head of standard attention, in the page's order, and the
    byte model built on them: 4 N d (Q, K, V, O once) + 4 N^2 (S and P each written and read)."""
    sys.path.insert(0, ROOT)
    import bench
    g = _read_keys("page_numbers.txt")
    accesses = tuple(a.strip() for a in g["standard_hbm_accesses"].split(","))
    assert len(accesses) == int(g["standard_hbm_access_count"])
    assert bench.STANDARD_ATTENTION_HBM_ACCESSES == accesses
    for n, d, e in [(1, 1, 1), (1024, 128, 2), (4096, 64, 4)]:
        assert bench.standard_attention_hbm_bytes(n, d, e) == (4 * n * n + 4 * n * d) * e


def _read_arrays():
    out = {}
    with open(os.path.join(GOLDEN, "oracle_tiny.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, *vals = line.split()
            out[name] = np.array([float(v) for v in vals])
    return out


@pytest.fixture(scope="module")
def stored():
    return _read_arrays()


def test_oracle_matches_its_stored_outputs(stored):
    sys.path.insert(0, GOLDEN)
    import make_oracle_tiny
    now = make_oracle_tiny.compute()
    assert set(now) == set(stored)
    for name, arr in now.items():
        np.testing.assert_allclose(arr, stored[name], rtol=1e-13, atol=1e-15, err_msg=name)


def test_stored_causal_first_row_is_the_first_value_row(stored):
    """Independent of the oracle: under the causal mask query 0 sees key 0 only, so its output
    is V's first row exactly and its LSE is scale <q_0, k_0>; its dQ is zero."""
    sys.path.insert(0, GOLDEN)
    import make_oracle_tiny
    from io_aware_attention_fa2_gb300.inputs import make_qkv
    c = make_oracle_tiny.CASE
    B, H, N, d = c["B"], c["H"], c["N"], c["d"]
    qb, kb, vb = make_qkv(B, H, N, d, c["dtype"], c["seed"])
    import oracle
    q, k, v = (oracle.decode(x, c["dtype"]) for x in (qb, kb, vb))
    o = stored["o_causal"].reshape(B, N, H, d)
    lse = stored["lse_causal"].reshape(B, H, N)
    dq = stored["dq_causal"].reshape(B, N, H, d)
    for b in range(B):
        for h in range(H):
            assert np.array_equal(o[b, 0, h], v[b, 0, h])
            assert lse[b, h, 0] == pytest.approx(c["scale"] * float(q[b, 0, h] @ k[b, 0, h]),
                                                 rel=1e-15, abs=1e-15)
            assert not dq[b, 0, h].any()
