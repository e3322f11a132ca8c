"""Pins for the oracle's alternative weight kernels (the ablation of reply A3
"Justification for Euclidean Distance Claim" in the OpenReview discussion of
"ZETA: Leveraging Z-order Curves for Efficient Top-k Attention": Cauchy softmax
against negative Euclidean with the usual softmax, and inverse Euclidean).

Readings: softmax of the logits -|q - k|^2 / gamma^2 over the attended set
(rowsum reported with the row's smallest squared distance as shift); inverse
Euclidean w = 1 / sqrt(|q - k|^2 + 1e-12).
"""
import numpy as np
import pytest
from scipy.special import softmax

from order_retrieval_gb300 import workloads as W

SOFTMAX, INV = 1, 2


def _inputs(seed, N, d_K=3, d_V=8):
    rng = np.random.default_rng(seed)
    q = rng.uniform(-1, 1, size=(N, d_K)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, d_K)).astype(np.float32)
    v = rng.normal(size=(N, d_V))
    return q, kx, v


def _sel(oracle_mod, q, kx, C, k):
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    return oracle_mod.select(qc[None], kc[None], C, k)[0]


def _set(idx_row, i, C):
    return [j for j in idx_row if j >= 0] + list(range((i // C) * C, i + 1))


@pytest.mark.parametrize("gamma", [0.05, 0.5, 2.0])
def test_softmax_full_window_is_scipy_softmax(oracle_mod, gamma):
    """Every key attended: dense causal softmax of -D^2 / gamma^2 (scipy)."""
    N, C = 64, 16
    q, kx, v = _inputs(41, N)
    idx = _sel(oracle_mod, q, kx, C, N)
    out, s = oracle_mod.attend_fwd(q, kx, v, gamma, idx, C, kind=SOFTMAX)
    d2 = ((q[:, None, :].astype(np.float64) - kx[None].astype(np.float64)) ** 2).sum(-1)
    logits = np.where(np.tril(np.ones((N, N), bool)), -d2 / gamma ** 2, -np.inf)
    a = softmax(logits, axis=1)
    np.testing.assert_allclose(out, a @ v, rtol=0, atol=1e-12)
    # rowsum = sum_j exp(logit_j - max logit): at least 1, and the largest weight is 1
    assert (s >= 1.0).all()
    np.testing.assert_allclose(s, 1.0 / a.max(1), rtol=1e-12)


def test_softmax_limits(oracle_mod):
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(42, N)
    idx = _sel(oracle_mod, q, kx, C, k)
    # gamma -> 0: all weight on the nearest key (no underflow thanks to the shift)
    o0, s0 = oracle_mod.attend_fwd(q, kx, v, 1e-4, idx, C, kind=SOFTMAX)
    # gamma -> infinity: uniform mean
    oi, si = oracle_mod.attend_fwd(q, kx, v, 1e6, idx, C, kind=SOFTMAX)
    for i in range(N):
        sel = _set(idx[i], i, C)
        d2 = ((q[i].astype(np.float64) - kx[sel].astype(np.float64)) ** 2).sum(1)
        np.testing.assert_allclose(o0[i], v[sel[int(np.argmin(d2))]], rtol=0, atol=1e-12)
        assert abs(s0[i] - 1.0) < 1e-12
        np.testing.assert_allclose(oi[i], v[sel].mean(0), rtol=0, atol=1e-9)
        np.testing.assert_allclose(si[i], len(sel), rtol=1e-9)


def test_inverse_euclidean_hand_example(oracle_mod):
    """One chunk of three tokens; query 2 at the origin sees keys at distances
    1, 2 and 4: weights 1, 1/2, 1/4, so a = (4/7, 2/7, 1/7)."""
    q = np.zeros((3, 3), np.float32)
    kx = np.array([[1, 0, 0], [0, 2, 0], [0, 0, 4]], np.float32)
    v = np.array([[7.0], [0.0], [0.0]])
    idx = np.full((3, 1), -1, np.int32)
    out, s = oracle_mod.attend_fwd(q, kx, v, 0.5, idx, 3, kind=INV)
    assert abs(out[2, 0] - 4.0) < 1e-10
    assert abs(s[2] - 1.75) < 1e-10
    assert abs(out[0, 0] - 7.0) < 1e-12        # query 0 sees key 0 only


def test_inverse_euclidean_ignores_scale_and_gamma(oracle_mod):
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(43, N)
    idx = _sel(oracle_mod, q, kx, C, k)
    o1, _ = oracle_mod.attend_fwd(q, kx, v, 0.5, idx, C, kind=INV)
    o2, _ = oracle_mod.attend_fwd(q.astype(np.float64) * 3, kx.astype(np.float64) * 3, v, 7.0,
                                  idx, C, kind=INV)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-9)
    # A query sitting on one of its keys takes (almost) that key's value.
    q2 = q.copy()
    q2[40] = kx[38]
    o3, _ = oracle_mod.attend_fwd(q2, kx, v, 0.5, idx, C, kind=INV)
    np.testing.assert_allclose(o3[40], v[38], rtol=0, atol=1e-4)


@pytest.mark.parametrize("kind", [SOFTMAX, INV])
def test_translation_and_constant_values(oracle_mod, kind):
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(44, N)
    idx = _sel(oracle_mod, q, kx, C, k)
    o1, s1 = oracle_mod.attend_fwd(q, kx, v, 0.4, idx, C, kind=kind)
    t = np.array([0.25, -0.5, 0.125])
    o2, s2 = oracle_mod.attend_fwd(q.astype(np.float64) + t, kx.astype(np.float64) + t, v, 0.4,
                                   idx, C, kind=kind)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-9)
    ones, _ = oracle_mod.attend_fwd(q, kx, np.ones((N, 3)), 0.4, idx, C, kind=kind)
    np.testing.assert_allclose(ones, 1.0, rtol=0, atol=1e-13)


def _loss(oracle_mod, q, kx, v, gamma, idx, dout, C, kind):
    out, _ = oracle_mod.attend_fwd(q, kx, v, gamma, idx, C, kind=kind)
    return float((out * dout).sum())


@pytest.mark.parametrize("kind", [SOFTMAX, INV])
def test_backward_matches_finite_differences(oracle_mod, kind):
    """Central differences in double, selection held fixed."""
    w = W.FD
    g = W.generate(w.replace(v_dtype="f32"), with_dout=True)
    q = g["q"][0, 0].astype(np.float64)
    kx = g["k"][0, 0].astype(np.float64)
    v = g["v"][0, 0].astype(np.float64)
    do = g["dout"][0, 0].astype(np.float64)
    gamma = float(g["gamma"][0])
    idx = _sel(oracle_mod, g["q"][0, 0], g["k"][0, 0], w.C, w.k)
    dq, dk, dv, dg = oracle_mod.attend_bwd(q, kx, v, gamma, idx, do, w.C, kind=kind)
    h = 1e-5 if kind == INV else 1e-4
    rng = np.random.default_rng(kind)
    for name, arr, grad in (("q", q, dq), ("kx", kx, dk), ("v", v, dv)):
        for _ in range(12):
            pos = tuple(rng.integers(0, s) for s in arr.shape)
            a, b = arr.copy(), arr.copy()
            a[pos] += h
            b[pos] -= h
            args_a = dict(q=q, kx=kx, v=v)
            args_b = dict(q=q, kx=kx, v=v)
            args_a[name], args_b[name] = a, b
            num = (_loss(oracle_mod, gamma=gamma, idx=idx, dout=do, C=w.C, kind=kind, **args_a)
                   - _loss(oracle_mod, gamma=gamma, idx=idx, dout=do, C=w.C, kind=kind,
                           **args_b)) / (2 * h)
            assert abs(num - grad[pos]) <= 1e-5 * max(1.0, abs(grad[pos])), (name, pos)
    num = (_loss(oracle_mod, q, kx, v, gamma + 1e-4, idx, do, w.C, kind)
           - _loss(oracle_mod, q, kx, v, gamma - 1e-4, idx, do, w.C, kind)) / 2e-4
    assert abs(num - dg) <= 1e-6 * max(1.0, abs(dg))
    if kind == INV:
        assert dg == 0.0


@pytest.mark.parametrize("kind", [SOFTMAX, INV])
def test_backward_invariants(oracle_mod, kind):
    """Translation: sum dq + sum dk = 0; values: sum_j dv_j = sum_i dO_i;
    scale: sum q.dq + sum k.dk + gamma dgamma = 0 (softmax depends on q/gamma,
    k/gamma; inverse Euclidean on neither scale nor gamma)."""
    N, C, k = 96, 32, 8
    q, kx, v = _inputs(45, N, d_V=6)
    do = np.random.default_rng(46).normal(size=(N, 6))
    idx = _sel(oracle_mod, q, kx, C, k)
    gamma = 0.6
    dq, dk, dv, dg = oracle_mod.attend_bwd(q, kx, v, gamma, idx, do, C, kind=kind)
    np.testing.assert_allclose(dq.sum(0) + dk.sum(0), 0.0, atol=1e-9)
    np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=1e-11)
    scale = (q.astype(np.float64) * dq).sum() + (kx.astype(np.float64) * dk).sum() + gamma * dg
    assert abs(scale) < 1e-8 * max(1.0, np.abs(dq).sum())
