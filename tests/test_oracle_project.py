"""Pins for the oracle's two-layer projection (OpenReview discussion of "ZETA:
Leveraging Z-order Curves for Efficient Top-k Attention", reply A "LLMs impact
the selection of d_K": a two-layer network projects the input into keys).

Reading: per head, Linear(D -> F), ReLU, Linear(F -> d_K), tanh (coordinates in
(-1, 1), the quantiser's range)."""
import numpy as np


def _weights(rng, D, H, F, d_K):
    return (rng.normal(size=(H * F, D)), rng.normal(size=H * F), rng.normal(size=(H, d_K, F)),
            rng.normal(size=(H, d_K)))


def test_selector_weights_give_closed_forms(oracle_mod):
    """W1 picks input e(hd, f) for hidden unit f; W2 picks hidden unit c for
    output c: y_c = tanh(max(0, x[e] + b1) + b2)."""
    rng = np.random.default_rng(60)
    M, D, H, F, d_K = 7, 11, 2, 4, 3
    x = rng.normal(size=(M, D))
    W1 = np.zeros((H * F, D))
    pick = rng.integers(0, D, size=H * F)
    W1[np.arange(H * F), pick] = 1.0
    b1 = rng.normal(size=H * F)
    W2 = np.zeros((H, d_K, F))
    for hd in range(H):
        for c in range(d_K):
            W2[hd, c, c + 1] = 1.0
    b2 = rng.normal(size=(H, d_K))
    out = oracle_mod.project(x, W1, b1, W2, b2)
    for t in range(M):
        for hd in range(H):
            for c in range(d_K):
                u = hd * F + c + 1
                want = np.tanh(max(0.0, x[t, pick[u]] + b1[u]) + b2[hd, c])
                assert abs(out[t, hd, c] - want) < 1e-15


def test_zero_first_layer_and_bias_only(oracle_mod):
    rng = np.random.default_rng(61)
    M, D, H, F, d_K = 5, 8, 3, 6, 3
    x = rng.normal(size=(M, D))
    W1, b1, W2, b2 = _weights(rng, D, H, F, d_K)
    out = oracle_mod.project(x, np.zeros_like(W1), b1, W2, b2)
    for hd in range(H):
        h = np.maximum(b1[hd * F:(hd + 1) * F], 0.0)
        for c in range(d_K):
            np.testing.assert_allclose(out[:, hd, c], np.tanh(W2[hd, c] @ h + b2[hd, c]),
                                       rtol=0, atol=1e-14)


def test_positive_homogeneity_without_biases(oracle_mod):
    """With zero biases, relu is positively homogeneous: atanh y(a x) = a atanh y(x)."""
    rng = np.random.default_rng(62)
    M, D, H, F, d_K = 6, 16, 2, 8, 3
    x = rng.normal(size=(M, D)) * 0.1
    W1, _, W2, _ = _weights(rng, D, H, F, d_K)
    W2 *= 0.1
    z1, z2 = np.zeros(H * F), np.zeros((H, d_K))
    y1 = oracle_mod.project(x, W1, z1, W2, z2)
    y3 = oracle_mod.project(3.0 * x, W1, z1, W2, z2)
    np.testing.assert_allclose(np.arctanh(y3), 3.0 * np.arctanh(y1), rtol=1e-12, atol=1e-14)


def test_heads_are_independent_and_ordered(oracle_mod):
    """Head hd reads rows hd*F..hd*F+F-1 of W1 only: changing another head's
    rows leaves it unchanged; swapping two heads' weights swaps the outputs."""
    rng = np.random.default_rng(63)
    M, D, H, F, d_K = 4, 10, 3, 5, 3
    x = rng.normal(size=(M, D))
    W1, b1, W2, b2 = _weights(rng, D, H, F, d_K)
    base = oracle_mod.project(x, W1, b1, W2, b2)
    W1b = W1.copy()
    W1b[F:2 * F] += 1.0
    other = oracle_mod.project(x, W1b, b1, W2, b2)
    assert np.array_equal(base[:, 0], other[:, 0]) and np.array_equal(base[:, 2], other[:, 2])
    assert not np.allclose(base[:, 1], other[:, 1])
    perm = [2, 0, 1]
    W1p = np.concatenate([W1[h * F:(h + 1) * F] for h in perm])
    b1p = np.concatenate([b1[h * F:(h + 1) * F] for h in perm])
    sw = oracle_mod.project(x, W1p, b1p, W2[perm], b2[perm])
    np.testing.assert_allclose(sw, base[:, perm], rtol=0, atol=1e-15)
