"""Pins for the multi-curve oracle functions (axis-permuted codes, the union of
per-curve windows).

Source: "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention",
OpenReview discussion, follow-up reply on interleaving the bits of
different dimensions (several curves): three curves
over the cyclic shifts of (K^1, K^2, K^3), or six over all orderings, each
contributing k//3 (k//6) of the k selected tokens.

Reading taken for the union: windows are listed in curve order, a token that
an earlier curve already contributed is dropped, and the row is filled to k
with -1 (no key).
"""
import bisect

import numpy as np
import pytest


def _bits_code(u, bits):
    """Morton code by an explicit bit loop: level j (from the top) emits the
    bit of every coordinate in slot order."""
    code = 0
    for j in reversed(range(bits)):
        for x in u:
            code = (code << 1) | ((int(x) >> j) & 1)
    return code


def test_encode_axes_is_a_column_permutation(oracle_mod):
    rng = np.random.default_rng(21)
    x = rng.uniform(-1, 1, size=(200, 3)).astype(np.float32)
    for axes in ([0, 1, 2], [1, 2, 0], [2, 0, 1], [0, 2, 1], [1, 0, 2], [2, 1, 0]):
        got = oracle_mod.encode_axes(x, 10, axes)
        want = oracle_mod.encode(np.ascontiguousarray(x[:, axes]), 10)
        assert np.array_equal(got, want)


@pytest.mark.parametrize("bits", [3, 12])
def test_encode_axes_bit_loop(oracle_mod, bits):
    rng = np.random.default_rng(22 + bits)
    x = rng.uniform(-1, 1, size=(50, 3)).astype(np.float32)
    u = np.array([[oracle_mod.quantise(float(v), bits) for v in r] for r in x])
    for axes in ([1, 2, 0], [2, 1, 0]):
        got = oracle_mod.encode_axes(x, bits, axes)
        for t in range(len(x)):
            assert int(got[t]) == _bits_code(u[t, axes], bits)


def test_curve_orders_are_the_pages_orders(oracle_mod):
    # Three curves: the cyclic shifts; six: every ordering exactly once.
    three = oracle_mod.curve_axes(3, 3)
    assert three == [[0, 1, 2], [1, 2, 0], [2, 0, 1]]
    six = oracle_mod.curve_axes(3, 6)
    assert sorted(map(tuple, six)) == sorted(
        (a, b, c) for a in range(3) for b in range(3) for c in range(3)
        if len({a, b, c}) == 3)
    assert six[0] == [0, 1, 2] and six[2] == [1, 2, 0] and six[4] == [2, 0, 1]
    assert oracle_mod.curve_axes(5, 1) == [[0, 1, 2, 3, 4]]


def test_merge_windows_hand_example(oracle_mod):
    w = np.array([[[1, 2, 3], [3, 4, -1], [2, 5, 6]]], dtype=np.int32)
    assert oracle_mod.merge_windows(w, 7)[0].tolist() == [1, 2, 3, 4, 5, 6, -1]
    assert oracle_mod.merge_windows(w, 9)[0].tolist() == [1, 2, 3, 4, 5, 6, -1, -1, -1]


def test_merge_windows_matches_ordered_set(oracle_mod):
    rng = np.random.default_rng(23)
    for M, km in ((3, 5), (6, 4), (2, 16)):
        w = rng.integers(-1, 12, size=(40, M, km)).astype(np.int32)
        got = oracle_mod.merge_windows(w, M * km + 2)
        for r in range(w.shape[0]):
            seen = list(dict.fromkeys(int(j) for j in w[r].reshape(-1) if j >= 0))
            assert got[r].tolist() == seen + [-1] * (M * km + 2 - len(seen))


def _brute_curve_window(q_code, i, kc, C, km):
    """One curve's window by brute force (same rule as the single curve)."""
    M = (i // C) * C
    pairs = sorted((int(kc[j]), j) for j in range(M))
    r = bisect.bisect_left(pairs, (int(q_code), i))
    order = sorted(sorted(range(M), key=lambda p: (abs(p - (r - 0.5)), p))[:km])
    return [pairs[p][1] for p in order]


@pytest.mark.parametrize("curves,k", [(3, 12), (6, 12), (3, 8), (6, 16)])
def test_select_multi_matches_brute_force(oracle_mod, curves, k):
    rng = np.random.default_rng(30 + curves + k)
    N, C = 64, 16
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    got = oracle_mod.select_multi(q, kx, C, k, 6, curves)
    km = k // curves
    u_q = np.array([[oracle_mod.quantise(float(v), 6) for v in r] for r in q])
    u_k = np.array([[oracle_mod.quantise(float(v), 6) for v in r] for r in kx])
    for i in range(N):
        if i < C:
            assert (got[i] == -1).all()
            continue
        seen = []
        for axes in oracle_mod.curve_axes(3, curves):
            kc = [_bits_code(u_k[j, axes], 6) for j in range(N)]
            seen += _brute_curve_window(_bits_code(u_q[i, axes], 6), i, kc, C, km)
        seen = list(dict.fromkeys(seen))
        assert got[i].tolist() == seen + [-1] * (k - len(seen))


def test_select_multi_one_curve_is_select(oracle_mod):
    rng = np.random.default_rng(31)
    N, C, k = 128, 32, 8
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    one = oracle_mod.select_multi(q, kx, C, k, 10, 1)
    ref = oracle_mod.select(oracle_mod.encode(q, 10)[None], oracle_mod.encode(kx, 10)[None],
                            C, k)[0]
    assert np.array_equal(one, ref)


@pytest.mark.parametrize("curves", [3, 6])
def test_select_multi_set_is_invariant_under_axis_relabelling(oracle_mod, curves):
    """The orders form a group (all orderings) or a coset-closed set (the cyclic
    shifts), so relabelling the axes of q and k by a member of that group gives
    the same SET of selected keys per query."""
    rng = np.random.default_rng(32 + curves)
    N, C, k = 96, 16, 12
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    base = oracle_mod.select_multi(q, kx, C, k, 8, curves)
    for pi in ([1, 2, 0], [2, 0, 1]) + (([0, 2, 1], [2, 1, 0]) if curves == 6 else ()):
        q2 = np.ascontiguousarray(q[:, pi])
        k2 = np.ascontiguousarray(kx[:, pi])
        rel = oracle_mod.select_multi(q2, k2, C, k, 8, curves)
        for i in range(N):
            assert set(base[i].tolist()) == set(rel[i].tolist())


def test_select_multi_invariants(oracle_mod):
    rng = np.random.default_rng(33)
    N, C, k = 128, 32, 16
    q = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    kx = rng.uniform(-1, 1, size=(N, 3)).astype(np.float32)
    for curves in (3, 6):
        got = oracle_mod.select_multi(q, kx, C, k, 10, curves)
        km = k // curves
        for i in range(C, N):
            row = [j for j in got[i].tolist() if j >= 0]
            assert len(row) == len(set(row))                        # no repeats
            assert km <= len(row) <= curves * km                    # first curve whole
            assert all(0 <= j < (i // C) * C for j in row)          # causal
            assert (got[i, len(row):] == -1).all()                  # padding at the end
