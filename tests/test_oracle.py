"""Pins for the fp64 attention oracle, each independent of the oracle's own formulas.

* central finite differences of L = sum(O * dO) (gradients vs the forward);
* scipy's softmax / logsumexp on the masked score matrix (forward vs a library routine);
* a two-key closed form (forward scale and sign);
* shift invariance of the keys: sum over keys of dK is zero (the D = rowsum(dO*O) term);
* causal brute force: row i equals a full-mask problem over keys 0..i;
* special cases: s = 1, and Q = 0 (uniform attention).
"""

import numpy as np
import pytest
import scipy.special

from oracle.attention import attn_bwd, attn_bwd_slice, attn_fwd, attn_fwd_slice


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss(q, k, v, do, scale, causal):
    o, _ = attn_fwd_slice(q, k, v, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("d", [2, 4])
def test_finite_differences(s, d, causal):
    rng = np.random.default_rng(100 * s + d + causal)
    q, k, v, do = (_rand(rng, s, d) for _ in range(4))
    scale = 1.0 / np.sqrt(d) * 1.7
    o, lse = attn_fwd_slice(q, k, v, scale, causal)
    dq, dk, dv = attn_bwd_slice(q, k, v, o, do, lse, scale, causal)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, do, scale, causal)
            x[idx] = old - eps
            lm = _loss(q, k, v, do, scale, causal)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        denom = max(np.abs(fd).max(), 1e-3)
        assert np.abs(fd - g).max() / denom <= 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_scipy_softmax(causal):
    rng = np.random.default_rng(7)
    s, d = 37, 16
    q, k, v = (_rand(rng, s, d) for _ in range(3))
    scale = 0.3
    logits = scale * np.einsum("id,jd->ij", q, k)
    if causal:
        logits = np.where(np.tril(np.ones((s, s), dtype=bool)), logits, -np.inf)
    o, lse = attn_fwd_slice(q, k, v, scale, causal, row_block=5)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(logits, axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, scipy.special.softmax(logits, axis=1) @ v, rtol=0, atol=1e-12)


def test_two_key_closed_form():
    # One query, two keys: O = sigmoid(scale * q.(k0 - k1)) v0 + sigmoid(scale * q.(k1 - k0)) v1.
    q = np.array([[0.5, -1.0, 2.0]])
    k = np.array([[1.0, 0.0, 0.5], [-0.5, 1.0, 0.0]])
    v = np.array([[1.0, 2.0, 3.0], [-4.0, 5.0, 0.25]])
    scale = 0.75
    # q.k0 = 0.5 + 0 + 1 = 1.5 ; q.k1 = -0.25 - 1 + 0 = -1.25
    z = scale * (1.5 - (-1.25))
    w0 = 1.0 / (1.0 + np.exp(-z))
    qq = np.vstack([q, q])      # second query row so the full mask sees both keys
    o, lse = attn_fwd_slice(qq, k, v, scale, causal=False)
    np.testing.assert_allclose(o[0], w0 * v[0] + (1 - w0) * v[1], rtol=1e-14)
    np.testing.assert_allclose(lse[0], np.log(np.exp(scale * 1.5) + np.exp(scale * -1.25)), rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance_and_dk_row_sum(causal):
    # Adding one vector to every key shifts each score row by a constant: P, O, dV, dQ
    # unchanged. Hence sum over keys of dK = scale * sum_i (sum_j dS_ij) Q_i = 0, which
    # holds only when dS = P * (dP - D) uses D = rowsum(dO * O).
    rng = np.random.default_rng(3)
    s, d = 24, 8
    q, k, v, do = (_rand(rng, s, d) for _ in range(4))
    scale = 1 / np.sqrt(d)
    o, lse = attn_fwd_slice(q, k, v, scale, causal)
    dq, dk, dv = attn_bwd_slice(q, k, v, o, do, lse, scale, causal)
    assert np.abs(dk.sum(axis=0)).max() <= 1e-12 * np.abs(dk).max() * s
    shift = _rand(rng, 1, d)
    o2, lse2 = attn_fwd_slice(q, k + shift, v, scale, causal)
    dq2, dk2, dv2 = attn_bwd_slice(q, k + shift, v, o2, do, lse2, scale, causal)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(dq2, dq, atol=1e-12)
    np.testing.assert_allclose(dk2, dk, atol=1e-12)
    np.testing.assert_allclose(dv2, dv, atol=1e-12)


def test_causal_brute_force_prefix():
    # Causal query row i is a full-mask problem over keys 0..i; dK/dV sum those.
    rng = np.random.default_rng(11)
    s, d = 13, 4
    q, k, v, do = (_rand(rng, s, d) for _ in range(4))
    scale = 0.6
    o, lse = attn_fwd_slice(q, k, v, scale, causal=True, row_block=4)
    dq, dk, dv = attn_bwd_slice(q, k, v, o, do, lse, scale, causal=True, row_block=4)
    dk_ref = np.zeros_like(k)
    dv_ref = np.zeros_like(v)
    for i in range(s):
        qi = q[i:i + 1]
        kp, vp = k[: i + 1], v[: i + 1]
        # full mask over the prefix: pad the single query up to the key count, one row only counts
        oi, lsei = attn_fwd_slice(np.repeat(qi, i + 1, axis=0), kp, vp, scale, causal=False)
        np.testing.assert_allclose(o[i], oi[0], atol=1e-12)
        np.testing.assert_allclose(lse[i], lsei[0], atol=1e-12)
        do_i = np.zeros((i + 1, d))
        do_i[0] = do[i]
        gq, gk, gv = attn_bwd_slice(np.repeat(qi, i + 1, axis=0), kp, vp, oi, do_i, lsei, scale, False)
        np.testing.assert_allclose(dq[i], gq[0], atol=1e-12)
        dk_ref[: i + 1] += gk
        dv_ref[: i + 1] += gv
    np.testing.assert_allclose(dk, dk_ref, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_single_token(causal):
    rng = np.random.default_rng(5)
    q, k, v, do = (_rand(rng, 1, 6) for _ in range(4))
    o, lse = attn_fwd_slice(q, k, v, 0.4, causal)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.4 * (q * k).sum(axis=1), atol=1e-15)
    dq, dk, dv = attn_bwd_slice(q, k, v, o, do, lse, 0.4, causal)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    assert np.abs(dq).max() <= 1e-15 and np.abs(dk).max() <= 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_uniform(causal):
    rng = np.random.default_rng(9)
    s, d = 10, 3
    q = np.zeros((s, d))
    k, v, do = (_rand(rng, s, d) for _ in range(3))
    o, lse = attn_fwd_slice(q, k, v, 0.5, causal)
    if causal:
        counts = np.arange(1, s + 1)[:, None]
        np.testing.assert_allclose(o, np.cumsum(v, axis=0) / counts, atol=1e-13)
        np.testing.assert_allclose(lse, np.log(np.arange(1, s + 1)), atol=1e-13)
        # dV_j = sum_{i >= j} dO_i / (i + 1)
        w = do / counts
        dv_ref = np.cumsum(w[::-1], axis=0)[::-1]
    else:
        np.testing.assert_allclose(o, np.repeat(v.mean(axis=0, keepdims=True), s, axis=0), atol=1e-13)
        np.testing.assert_allclose(lse, np.full(s, np.log(s)), atol=1e-13)
        dv_ref = np.repeat(do.sum(axis=0, keepdims=True) / s, s, axis=0)
    _, _, dv = attn_bwd_slice(q, k, v, o, do, lse, 0.5, causal)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-13)


def test_bshd_wrapper_and_head_subset():
    rng = np.random.default_rng(2)
    b, s, h, d = 2, 9, 3, 4
    q, k, v, do = (_rand(rng, b, s, h, d) for _ in range(4))
    o, lse = attn_fwd(q, k, v, 0.5, True)
    dq, dk, dv = attn_bwd(q, k, v, o, do, lse, 0.5, True, row_block=2)
    for bi in range(b):
        for hi in range(h):
            os_, ls_ = attn_fwd_slice(q[bi, :, hi], k[bi, :, hi], v[bi, :, hi], 0.5, True)
            np.testing.assert_allclose(o[bi, :, hi], os_)
            np.testing.assert_allclose(lse[bi, hi], ls_)
            g = attn_bwd_slice(q[bi, :, hi], k[bi, :, hi], v[bi, :, hi], os_, do[bi, :, hi], ls_, 0.5, True)
            np.testing.assert_allclose(dq[bi, :, hi], g[0], atol=1e-13)
            np.testing.assert_allclose(dk[bi, :, hi], g[1], atol=1e-13)
            np.testing.assert_allclose(dv[bi, :, hi], g[2], atol=1e-13)
    sub = attn_bwd(q, k, v, o, do, lse, 0.5, True, heads=[(1, 2)])
    assert np.isnan(sub[0][0]).all() and np.allclose(sub[0][1, :, 2], dq[1, :, 2])
