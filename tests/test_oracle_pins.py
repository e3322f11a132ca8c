"""Pins for the CPU oracle: each checks it against something other than itself.

Sources ("ZETA: Leveraging Z-order Curves for Efficient Top-k Attention"):
  - OpenReview discussion, reply A2 "Clarification of Binary Expansion and
    Precision": normalise each coordinate to [0, 1], discretise to a 4096-cell
    grid (12 bits), interleave the bits, result fits a 64-bit integer.
  - OpenReview discussion, reply A3 "Chunking ... & Where efficiency is coming
    from" and reply A2 "Clarification": radix sort of Z codes, binary search of
    the query's insertion position, the window centred there is the neighbour set.
  - OpenReview discussion, reply A2 "Discussion on its robustness": trainable
    gamma is a temperature; gamma = 1 gives a Student-t kernel.
"""
import bisect

import numpy as np
import pytest

from order_retrieval_gb300 import workloads as W


# ------------------------------------------------------------- quantiser ---

@pytest.mark.parametrize("bits", [1, 3, 10, 12, 21, 24])
def test_quantise_grid_points_and_cells(oracle_mod, bits):
    """x = -1 + m / 2^(bits-1) is the left edge of cell m; points inside the
    cell stay in it; the ends clamp (closed form of a uniform 2^bits grid on
    [-1, 1))."""
    half = 2.0 ** (bits - 1)
    cells = 2 ** bits
    ms = sorted({0, 1, cells // 3, cells // 2, cells - 2, cells - 1} & set(range(cells)))
    for m in ms:
        edge = np.float32(-1.0 + m / half)
        assert oracle_mod.quantise(float(edge), bits) == m
        inside = np.float32(-1.0 + (m + 0.5) / half)
        assert oracle_mod.quantise(float(inside), bits) == m
    assert oracle_mod.quantise(float(np.nextafter(np.float32(1), np.float32(0))), bits) == cells - 1
    assert oracle_mod.quantise(-1.0, bits) == 0
    assert oracle_mod.quantise(-3.5, bits) == 0
    assert oracle_mod.quantise(1.0, bits) == cells - 1
    assert oracle_mod.quantise(7.0, bits) == cells - 1
    assert oracle_mod.quantise(float("nan"), bits) == 0
    assert oracle_mod.quantise(float("inf"), bits) == cells - 1
    assert oracle_mod.quantise(float("-inf"), bits) == 0


def test_quantise_twelve_bit_grid_matches_pages(oracle_mod):
    """12 bits per coordinate: integers 0..4095 (OpenReview reply A2)."""
    xs = np.linspace(-1, 1, 9999, endpoint=False, dtype=np.float32)
    u = [oracle_mod.quantise(float(x), 12) for x in xs]
    assert min(u) == 0 and max(u) == 4095
    assert all(b >= a for a, b in zip(u, u[1:]))


# ------------------------------------------------------------ interleave ---

# Hand table for d_K = 3, bits = 10: a single set bit j of coordinate d lands at
# code bit 3*j + (2 - d) (level j, coordinate 0 most significant in a level).
SINGLE_BIT_D3 = [
    # (d, j, code)
    (0, 0, 4), (1, 0, 2), (2, 0, 1),
    (0, 1, 32), (1, 1, 16), (2, 1, 8),
    (0, 5, 1 << 17), (1, 5, 1 << 16), (2, 5, 1 << 15),
    (0, 9, 1 << 29), (1, 9, 1 << 28), (2, 9, 1 << 27),
]


@pytest.mark.parametrize("d,j,code", SINGLE_BIT_D3)
def test_interleave_single_bit_positions(oracle_mod, d, j, code):
    u = [0, 0, 0]
    u[d] = 1 << j
    assert oracle_mod.interleave(u, 10) == code


def test_interleave_hand_examples(oracle_mod):
    # u = (5, 3, 6) in 3 bits: levels from LSB: l0 = (1,1,0) -> 0b110, l1 = (0,1,1) -> 0b011,
    # l2 = (1,0,1) -> 0b101; code = 0b101_011_110 = 350.
    assert oracle_mod.interleave([5, 3, 6], 3) == 0b101011110
    # d_K = 2, u = (2, 1) in 2 bits: l0 = (0,1) -> 0b01, l1 = (1,0) -> 0b10 -> 0b1001 = 9.
    assert oracle_mod.interleave([2, 1], 2) == 9


@pytest.mark.parametrize("d_K,bits", [(1, 21), (2, 21), (3, 10), (3, 12), (8, 8)])
def test_interleave_extremes(oracle_mod, d_K, bits):
    assert oracle_mod.interleave([0] * d_K, bits) == 0
    assert oracle_mod.interleave([(1 << bits) - 1] * d_K, bits) == (1 << (d_K * bits)) - 1
    if d_K == 1:
        for u in (1, 12345, (1 << bits) - 2):
            assert oracle_mod.interleave([u], bits) == u


@pytest.mark.parametrize("d_K,bits", [(2, 6), (3, 5), (3, 10), (8, 8)])
def test_interleave_order_is_levelwise_lexicographic(oracle_mod, d_K, bits):
    """Z order = lexicographic order of the bit levels read from the most
    significant level down, coordinate 0 first in each level."""
    rng = np.random.default_rng(7)
    us = rng.integers(0, 1 << bits, size=(300, d_K))

    def levels(u):
        return tuple(int(u[d]) >> j & 1 for j in range(bits - 1, -1, -1) for d in range(d_K))

    codes = [oracle_mod.interleave(list(map(int, u)), bits) for u in us]
    keys = [levels(u) for u in us]
    by_code = sorted(range(len(us)), key=lambda t: (codes[t], t))
    by_levels = sorted(range(len(us)), key=lambda t: (keys[t], t))
    assert by_code == by_levels
    assert len(set(codes)) == len(set(keys))


def test_encode_matches_quantise_then_interleave_on_array(oracle_mod):
    rng = np.random.default_rng(3)
    x = rng.uniform(-1.2, 1.2, size=(50, 3)).astype(np.float32)
    codes = oracle_mod.encode(x, 10)
    for t in range(50):
        u = [oracle_mod.quantise(float(x[t, d]), 10) for d in range(3)]
        assert codes[t] == oracle_mod.interleave(u, 10)


# ------------------------------------------------------- sort and prefix ---

@pytest.mark.parametrize("bits", [1, 2, 10])
def test_prefix_table_equals_library_lexsort(oracle_mod, bits):
    """prefix_c = keys 0..cC-1 sorted by (code, index), checked against numpy's
    lexsort; heavy ties at low bit depth exercise the index tie-break."""
    rng = np.random.default_rng(bits)
    N, C = 96, 16
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kc = oracle_mod.encode(kx, bits)
    pc, pi = oracle_mod.prefix_table(kc[None], C)
    n = N // C
    assert pc.shape == (1, C * n * (n - 1) // 2)
    for c in range(1, n):
        off = C * c * (c - 1) // 2
        M = c * C
        want = np.lexsort((np.arange(M), kc[:M]))
        assert np.array_equal(pi[0, off:off + M], want)
        assert np.array_equal(pc[0, off:off + M], kc[want])
        assert sorted(pi[0, off:off + M].tolist()) == list(range(M))


# ---------------------------------------------------------------- select ---

def _brute_window(q_code, i, kc, C, k):
    """Window by brute force: insertion point of (code_q, i) among the sorted
    (code, index) pairs of the prefix, then the k positions nearest to the gap
    just before it, ties to the lower position."""
    c = i // C
    M = c * C
    pairs = sorted((int(kc[j]), j) for j in range(M))
    r = bisect.bisect_left(pairs, (int(q_code), i))
    order = sorted(range(M), key=lambda p: (abs(p - (r - 0.5)), p))[:k]
    order.sort()
    out = [pairs[p][1] for p in order]
    return out + [-1] * (k - len(out))


@pytest.mark.parametrize("k", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("bits", [2, 10])
def test_select_matches_brute_force(oracle_mod, k, bits):
    rng = np.random.default_rng(100 + k + bits)
    N, C = 64, 16
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    qc, kc = oracle_mod.encode(q, bits), oracle_mod.encode(kx, bits)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    for i in range(N):
        if i < C:
            assert (idx[i] == -1).all()
            continue
        assert idx[i].tolist() == _brute_window(qc[i], i, kc, C, k)


def test_select_invariants_and_full_prefix(oracle_mod):
    rng = np.random.default_rng(5)
    N, C, k = 128, 32, 8
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    for i in range(C, N):
        row = idx[i]
        assert len(set(row.tolist())) == k
        assert (row >= 0).all() and (row < (i // C) * C).all()     # causal
    # A window at least as long as every prefix selects the whole prefix.
    big = oracle_mod.select(qc[None], kc[None], C, N)[0]
    for i in range(C, N):
        M = (i // C) * C
        assert sorted(big[i, :M].tolist()) == list(range(M))
        assert (big[i, M:] == -1).all()


def test_select_rows_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(9)
    N, C, k = 96, 16, 4
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    full = oracle_mod.select(qc[None], kc[None], C, k)[0]
    rows = np.array([3, 17, 40, 41, 95])
    sub = oracle_mod.select(qc[None], kc[None], C, k, rows=rows)[0]
    assert np.array_equal(sub, full[rows])


# ---------------------------------------------------------------- attend ---

def _dense_causal_cauchy(q, kx, v, gamma):
    """Dense causal Cauchy attention in matrix form (float64)."""
    d2 = ((q[:, None, :] - kx[None, :, :]) ** 2).sum(-1)
    wm = 1.0 / (1.0 + d2 / gamma ** 2)
    wm = np.tril(wm)
    s = wm.sum(1)
    return (wm @ v) / s[:, None], s


def _inputs(seed, N, d_K=3, d_V=8):
    rng = np.random.default_rng(seed)
    q = rng.uniform(-1, 1, size=(N, d_K)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, d_K)).astype(np.float32)
    v = rng.normal(size=(N, d_V))
    return q, kx, v


@pytest.mark.parametrize("gamma", [0.3, 0.5, 1.0])
def test_attend_full_window_is_dense_causal(oracle_mod, gamma):
    """A window covering every prefix plus the own-chunk keys j <= i is exactly
    dense causal Cauchy attention."""
    N, C = 64, 16
    q, kx, v = _inputs(11, N)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, N)[0]
    out, s = oracle_mod.attend_fwd(q, kx, v, gamma, idx, C)
    ref, sref = _dense_causal_cauchy(q.astype(np.float64), kx.astype(np.float64), v, gamma)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s, sref, rtol=1e-13)


def test_attend_single_chunk_is_dense_causal(oracle_mod):
    N = 48
    q, kx, v = _inputs(12, N)
    idx = np.full((N, 4), -1, dtype=np.int32)
    out, _ = oracle_mod.attend_fwd(q, kx, v, 0.7, idx, N)
    ref, _ = _dense_causal_cauchy(q.astype(np.float64), kx.astype(np.float64), v, 0.7)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_attend_special_cases(oracle_mod):
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(13, N)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    # Weights are normalised: constant values pass through unchanged.
    ones = np.ones((N, 5))
    o1, _ = oracle_mod.attend_fwd(q, kx, ones, 0.5, idx, C)
    np.testing.assert_allclose(o1, 1.0, rtol=0, atol=1e-14)
    # gamma -> infinity: every selected key weighs the same (uniform mean).
    ob, sb = oracle_mod.attend_fwd(q, kx, v, 1e7, idx, C)
    for i in range(N):
        sel = [j for j in idx[i] if j >= 0] + list(range((i // C) * C, i + 1))
        np.testing.assert_allclose(ob[i], v[sel].mean(0), rtol=0, atol=1e-9)
        np.testing.assert_allclose(sb[i], len(sel), rtol=1e-9)
    # All keys equal to the query: every weight is 1.
    same = np.zeros_like(q)
    os_, ss = oracle_mod.attend_fwd(same, same, v, 0.5, idx, C)
    for i in range(N):
        sel = [j for j in idx[i] if j >= 0] + list(range((i // C) * C, i + 1))
        np.testing.assert_allclose(os_[i], v[sel].mean(0), rtol=0, atol=1e-12)
        assert ss[i] == len(sel)


def test_attend_gamma_is_a_length_scale(oracle_mod):
    """w depends on |q - k| / gamma only: scaling q, k and gamma together leaves
    the output unchanged; gamma = 1 is the Student-t kernel 1 / (1 + d^2)."""
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(14, N)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    o1, s1 = oracle_mod.attend_fwd(q, kx, v, 0.25, idx, C)
    o2, s2 = oracle_mod.attend_fwd(q.astype(np.float64) * 4, kx.astype(np.float64) * 4, v, 1.0,
                                   idx, C)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s1, s2, rtol=1e-12)
    i = 40
    sel = [j for j in idx[i] if j >= 0] + list(range(32, i + 1))
    d2 = ((q[i].astype(np.float64) * 4 - kx[sel].astype(np.float64) * 4) ** 2).sum(1)
    np.testing.assert_allclose(s2[i], (1.0 / (1.0 + d2)).sum(), rtol=1e-13)


def test_attend_rows_subset(oracle_mod):
    N, C, k = 64, 16, 6
    q, kx, v = _inputs(15, N)
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    full, sf = oracle_mod.attend_fwd(q, kx, v, 0.5, idx, C)
    rows = np.array([0, 15, 16, 63])
    sub, ss = oracle_mod.attend_fwd(q, kx, v, 0.5, idx[rows], C, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(ss, sf[rows])


# -------------------------------------------------------------- backward ---

def _loss(oracle_mod, q, kx, v, gamma, idx, dout, C):
    out, _ = oracle_mod.attend_fwd(q, kx, v, gamma, idx, C)
    return float((out * dout).sum())


def test_backward_matches_finite_differences(oracle_mod):
    """Central differences in double with the selection held fixed."""
    w = W.FD
    g = W.generate(w.replace(v_dtype="f32"), with_dout=True)
    q = g["q"][0, 0].astype(np.float64)
    kx = g["k"][0, 0].astype(np.float64)
    v = g["v"][0, 0].astype(np.float64)
    do = g["dout"][0, 0].astype(np.float64)
    gamma = float(g["gamma"][0])
    qc = oracle_mod.encode(g["q"][0, 0], w.bits)
    kc = oracle_mod.encode(g["k"][0, 0], w.bits)
    idx = oracle_mod.select(qc[None], kc[None], w.C, w.k)[0]
    dq, dk, dv, dg = oracle_mod.attend_bwd(q, kx, v, gamma, idx, do, w.C)
    h = 1e-4
    rng = np.random.default_rng(0)

    def fd(arr, pos):
        a = arr.copy(); a[pos] += h
        b = arr.copy(); b[pos] -= h
        return a, b

    for name, arr, grad in (("q", q, dq), ("k", kx, dk), ("v", v, dv)):
        for _ in range(12):
            pos = tuple(rng.integers(0, s) for s in arr.shape)
            a, b = fd(arr, pos)
            args_a = dict(q=q, kx=kx, v=v)
            args_b = dict(q=q, kx=kx, v=v)
            key = {"q": "q", "k": "kx", "v": "v"}[name]
            args_a[key] = a
            args_b[key] = b
            num = (_loss(oracle_mod, gamma=gamma, idx=idx, dout=do, C=w.C, **args_a)
                   - _loss(oracle_mod, gamma=gamma, idx=idx, dout=do, C=w.C, **args_b)) / (2 * h)
            assert abs(num - grad[pos]) <= 1e-6 * max(1.0, abs(grad[pos])), (name, pos)
    num = (_loss(oracle_mod, q, kx, v, gamma + h, idx, do, w.C)
           - _loss(oracle_mod, q, kx, v, gamma - h, idx, do, w.C)) / (2 * h)
    assert abs(num - dg) <= 1e-6 * max(1.0, abs(dg))


def test_backward_invariants(oracle_mod):
    """Translation: sum dq + sum dk = 0.  Scale: sum q.dq + sum k.dk + gamma dgamma
    = 0 (the output depends on q/gamma, k/gamma only).  Values: sum_j dv_j =
    sum_i dO_i (weights of each query sum to one)."""
    N, C, k = 96, 32, 8
    q, kx, v = _inputs(21, N, d_V=6)
    do = np.random.default_rng(22).normal(size=(N, 6))
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    gamma = 0.6
    dq, dk, dv, dg = oracle_mod.attend_bwd(q, kx, v, gamma, idx, do, C)
    np.testing.assert_allclose(dq.sum(0) + dk.sum(0), 0.0, atol=1e-11)
    scale = (q.astype(np.float64) * dq).sum() + (kx.astype(np.float64) * dk).sum() + gamma * dg
    assert abs(scale) < 1e-10
    np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=1e-11)


def test_backward_row_shares_sum_to_the_gradient(oracle_mod):
    """The gradients are sums over queries: the shares of a partition of the
    queries (each part listed in rows, with its idx rows) add up to the full
    backward, and a part's dq is zero outside its rows."""
    N, C, k = 128, 32, 8
    q, kx, v = _inputs(41, N, d_V=5)
    do = np.random.default_rng(42).normal(size=(N, 5))
    qc, kc = oracle_mod.encode(q, 10), oracle_mod.encode(kx, 10)
    idx = oracle_mod.select(qc[None], kc[None], C, k)[0]
    full = oracle_mod.attend_bwd(q, kx, v, 0.7, idx, do, C)
    perm = np.random.default_rng(43).permutation(N)
    parts = [np.sort(perm[:50]), np.sort(perm[50:90]), np.sort(perm[90:])]
    tot = [np.zeros_like(full[0]), np.zeros_like(full[1]), np.zeros_like(full[2]), 0.0]
    for rows in parts:
        dq, dk, dv, dg = oracle_mod.attend_bwd(q, kx, v, 0.7, idx[rows], do, C, rows=rows)
        outside = np.setdiff1d(np.arange(N), rows)
        assert (dq[outside] == 0).all()
        tot = [tot[0] + dq, tot[1] + dk, tot[2] + dv, tot[3] + dg]
    for a, b in zip(tot[:3], full[:3]):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    assert abs(tot[3] - full[3]) <= 1e-12 * max(1.0, abs(full[3]))


# ---------------------------------------------------------------- recall ---

def test_exact_topk_matches_lexsort(oracle_mod):
    N, C, k = 80, 16, 5
    q, kx, _ = _inputs(31, N)
    out = oracle_mod.exact_topk(q, kx, C, k)
    for i in range(N):
        M = (i // C) * C
        if M == 0:
            assert (out[i] == -1).all()
            continue
        d2 = ((q[i].astype(np.float64) - kx[:M].astype(np.float64)) ** 2).sum(1)
        want = np.lexsort((np.arange(M), d2))[:k]
        got = out[i][out[i] >= 0]
        assert got.tolist() == want[:len(got)].tolist()


# ------------------------------------------------------------- generators ---

def test_splitmix64_published_value():
    """First SplitMix64 output for seed 0 (Steele, Lea, Flood 2014)."""
    assert int(W.SplitMix64(0).raw(1)[0]) == 0xE220A8397B1DCDAF


def test_generators_are_deterministic_and_in_range():
    a = W.generate(W.TINY)
    b = W.generate(W.TINY)
    for key in a:
        assert np.array_equal(a[key], b[key])
    assert a["q"].min() >= -1 and a["q"].max() < 1
    c = W.generate(W.CLUSTERED)
    assert c["q"].min() >= -1 and c["q"].max() < 1
    assert (c["gamma"] >= 0.3).all() and (c["gamma"] <= 1.0).all()
    widened = W.bf16_bits_to_f32(c["v"])
    assert np.abs(widened - c["v_f32"]).max() <= 2.0 ** -8 * np.abs(c["v_f32"]).max()
