"""Pins for the split-K GEMM oracle (oracle/gemm.py) that do not re-type its formula:
a brute-force triple loop on tiny inputs, the identity and transposition laws, and that
the chunk partials of any even split of K sum to the whole product."""
import numpy as np
import pytest

from oracle.gemm import gemm_nt, gemm_nt_split_partials


def test_brute_force_triple_loop():
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal((3, 5)), rng.standard_normal((4, 5))
    c = gemm_nt(a, b)
    for m in range(3):
        for n in range(4):
            s = 0.0
            for k in range(5):
                s += a[m, k] * b[n, k]
            assert c[m, n] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_identity_and_transpose():
    rng = np.random.default_rng(4)
    a = rng.standard_normal((6, 6))
    assert np.allclose(gemm_nt(a, np.eye(6)), a)                  # A I^T = A
    b = rng.standard_normal((5, 6))
    assert np.allclose(gemm_nt(a, b), gemm_nt(b, a).T)            # (A B^T)^T = B A^T


@pytest.mark.parametrize("splits", [1, 2, 3, 6])
def test_split_partials_sum_to_the_product(splits):
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((4, 12)), rng.standard_normal((7, 12))
    parts = gemm_nt_split_partials(a, b, splits)
    assert len(parts) == splits
    assert np.allclose(sum(parts), gemm_nt(a, b), rtol=1e-13, atol=1e-13)
    with pytest.raises(ValueError):
        gemm_nt_split_partials(a, b, 5)
