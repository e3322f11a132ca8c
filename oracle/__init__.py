"""CPU oracle for the ZETA hot path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product library never calls it and shares no code
with it.  The arithmetic lives in ``zeta_oracle.c`` (plain C, single-threaded,
double precision except the float32 quantiser); this module only builds it,
loads it and marshals numpy arrays, one (b, h) slice at a time.

Method: "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention"
(arXiv 2501.14577).  Each C function cites the passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zeta_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile zeta_oracle.c with gcc into liboracle.so next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    D = ctypes.c_double
    lib.orc_quantise.argtypes = [ctypes.c_float, I]
    lib.orc_quantise.restype = ctypes.c_uint32
    lib.orc_interleave.argtypes = [P, I, I]
    lib.orc_interleave.restype = ctypes.c_uint64
    lib.orc_encode.argtypes = [P, I64, I, I, P]
    lib.orc_prefix.argtypes = [P, I64, I64, P, P]
    lib.orc_prefix_table.argtypes = [P, I64, I64, P, P]
    lib.orc_select.argtypes = [P, P, I64, I64, I, P, I64, P]
    lib.orc_attend_fwd.argtypes = [P, P, P, D, P, I64, I64, I, I, I, P, I64, P, P, I]
    lib.orc_attend_bwd.argtypes = [P, P, P, D, P, P, I64, I64, I, I, I, P, P, P, P, I]
    lib.orc_attend_bwd_rows.argtypes = [P, P, P, D, P, P, I64, I64, I, I, I, P, I64,
                                        P, P, P, P, I]
    lib.orc_exact_topk.argtypes = [P, P, I64, I64, I, I, P, I64, P]
    lib.orc_encode_axes.argtypes = [P, I64, I, I, P, P]
    lib.orc_project.argtypes = [P, I64, I, I, I, I, P, P, P, P, P]
    lib.orc_merge_windows.argtypes = [P, I, I, I, P]
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, len(r)


# ----------------------------------------------------------------- encode ---

def quantise(x: float, bits: int) -> int:
    """Grid cell of one coordinate (float32 arithmetic)."""
    return int(_load().orc_quantise(ctypes.c_float(x), bits))


def interleave(u, bits: int) -> int:
    """Z-order code of one tuple of cell indices."""
    a = np.ascontiguousarray(u, dtype=np.uint32)
    return int(_load().orc_interleave(_p(a), len(a), bits))


def encode(x: np.ndarray, bits: int) -> np.ndarray:
    """x float32 [..., d_K] -> uint64 codes [...]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d_K = x.shape[-1]
    out = np.empty(x.shape[:-1], dtype=np.uint64)
    _load().orc_encode(_p(x), out.size, d_K, bits, _p(out))
    return out


def encode_axes(x: np.ndarray, bits: int, axes) -> np.ndarray:
    """Codes of the coordinates taken in the order `axes` (a permutation)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d_K = x.shape[-1]
    ax = np.ascontiguousarray(axes, dtype=np.int32)
    assert sorted(ax.tolist()) == list(range(d_K))
    out = np.empty(x.shape[:-1], dtype=np.uint64)
    _load().orc_encode_axes(_p(x), out.size, d_K, bits, _p(ax), _p(out))
    return out


def curve_axes(d_K: int, curves: int):
    """Axis orders of the multi-curve variant: 1 curve = identity; 3 curves =
    the cyclic shifts (0,1,2), (1,2,0), (2,0,1); 6 curves = all permutations in
    the pages' order (0,1,2), (0,2,1), (1,2,0), (1,0,2), (2,0,1), (2,1,0)."""
    if curves == 1:
        return [list(range(d_K))]
    assert d_K == 3, "multi-curve orders are defined for d_K = 3"
    if curves == 3:
        return [[0, 1, 2], [1, 2, 0], [2, 0, 1]]
    if curves == 6:
        return [[0, 1, 2], [0, 2, 1], [1, 2, 0], [1, 0, 2], [2, 0, 1], [2, 1, 0]]
    raise ValueError("curves must be 1, 3 or 6")


def merge_windows(windows: np.ndarray, k: int) -> np.ndarray:
    """windows int32 [..., M, km] -> union rows int32 [..., k] (curve order,
    first occurrence kept, -1 padded)."""
    w = np.ascontiguousarray(windows, dtype=np.int32)
    M, km = w.shape[-2], w.shape[-1]
    lead = w.shape[:-2]
    flat = w.reshape(-1, M * km)
    out = np.empty((flat.shape[0], k), dtype=np.int32)
    lib = _load()
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        o = out[r]
        lib.orc_merge_windows(_p(row), M, km, k, _p(o))
    return out.reshape(*lead, k)


def select_multi(q, kx, C: int, k: int, bits: int, curves: int, rows=None):
    """Multi-curve window of one slice: per curve, codes of the permuted axes,
    a window of k // curves keys; the union row of k entries."""
    km = k // curves
    wins = []
    for axes in curve_axes(q.shape[-1], curves):
        qc = encode_axes(q, bits, axes)
        kc = encode_axes(kx, bits, axes)
        wins.append(select(qc[None], kc[None], C, km, rows=rows)[0])
    return merge_windows(np.stack(wins, axis=-2), k)


def project(x, W1, b1, W2, b2):
    """Two-layer projection (see orc_project).  x [M, D]; W1 [H*F, D]; b1 [H*F];
    W2 [H, d_K, F]; b2 [H, d_K]; all taken as float64.  Returns [M, H, d_K]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W1 = np.ascontiguousarray(W1, dtype=np.float64)
    b1 = np.ascontiguousarray(b1, dtype=np.float64)
    W2 = np.ascontiguousarray(W2, dtype=np.float64)
    b2 = np.ascontiguousarray(b2, dtype=np.float64)
    M, D = x.shape
    H, d_K, F = W2.shape
    assert W1.shape == (H * F, D) and b1.shape == (H * F,) and b2.shape == (H, d_K)
    out = np.empty((M, H, d_K), dtype=np.float64)
    _load().orc_project(_p(x), M, D, H, F, d_K, _p(W1), _p(b1), _p(W2), _p(b2), _p(out))
    return out


# ------------------------------------------------------------ sort/select ---

def prefix_table(key_codes: np.ndarray, C: int):
    """key_codes uint64 [..., N] -> (codes uint64 [..., T], idx int32 [..., T])."""
    kc = np.ascontiguousarray(key_codes, dtype=np.uint64)
    N = kc.shape[-1]
    n = N // C
    T = C * n * (n - 1) // 2
    lead = kc.shape[:-1]
    flat = kc.reshape(-1, N)
    pc = np.zeros((flat.shape[0], T), dtype=np.uint64)
    pi = np.zeros((flat.shape[0], T), dtype=np.int32)
    lib = _load()
    for s in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[s])
        a, b = pc[s], pi[s]
        lib.orc_prefix_table(_p(row), N, C, _p(a), _p(b))
    return pc.reshape(*lead, T), pi.reshape(*lead, T)


def select(q_codes: np.ndarray, key_codes: np.ndarray, C: int, k: int, rows=None):
    """Top-k window indices.  q_codes/key_codes uint64 [S, N] (S slices).

    rows None: int32 [S, N, k].  rows given (1-D query list shared by all
    slices): int32 [S, len(rows), k]."""
    qc = np.ascontiguousarray(q_codes, dtype=np.uint64)
    kc = np.ascontiguousarray(key_codes, dtype=np.uint64)
    S, N = qc.shape
    r, nr = _rows(rows)
    cnt = nr if r is not None else N
    out = np.empty((S, cnt, k), dtype=np.int32)
    lib = _load()
    for s in range(S):
        a = np.ascontiguousarray(qc[s])
        b = np.ascontiguousarray(kc[s])
        o = out[s]
        lib.orc_select(_p(a), _p(b), N, C, k, _p(r) if r is not None else None, nr, _p(o))
    return out


# ----------------------------------------------------------------- attend ---

CAUCHY, SOFTMAX, INV_EUCLID = 0, 1, 2     # weight kernels (see zeta_oracle.c)


def attend_fwd(q, k, v, gamma: float, idx, C: int, rows=None, kind: int = CAUCHY):
    """One slice.  q,k [N,d_K]; v [N,d_V] (any float dtype, taken as double);
    idx int32 [R,k], one row per listed query (all N when rows is None).
    kind: CAUCHY, SOFTMAX (of -d2/gamma^2, rowsum taken with the row's
    smallest d2 as shift) or INV_EUCLID.
    Returns (out [R,d_V] float64, rowsum [R] float64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    kx = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, d_K = q.shape
    d_V = v.shape[1]
    kk = idx.shape[1]
    r, nr = _rows(rows)
    cnt = nr if r is not None else N
    out = np.empty((cnt, d_V), dtype=np.float64)
    rs = np.empty((cnt,), dtype=np.float64)
    _load().orc_attend_fwd(_p(q), _p(kx), _p(v), float(gamma), _p(idx), N, C, d_K, d_V, kk,
                           _p(r) if r is not None else None, nr, _p(out), _p(rs), int(kind))
    return out, rs


def attend_bwd(q, k, v, gamma: float, idx, dout, C: int, kind: int = CAUCHY, rows=None):
    """One slice, selection fixed.  Returns (dq, dk, dv, dgamma) in float64.

    rows None: the gradients (idx [N, k]).  rows given: only the listed
    queries contribute (idx holds their rows, [len(rows), k]); the results are
    their shares of the sums."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    kx = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    do = np.ascontiguousarray(dout, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, d_K = q.shape
    d_V = v.shape[1]
    kk = idx.shape[1]
    dq = np.empty_like(q)
    dk = np.empty_like(kx)
    dv = np.empty_like(v)
    dg = np.zeros(1, dtype=np.float64)
    r, nr = _rows(rows)
    _load().orc_attend_bwd_rows(_p(q), _p(kx), _p(v), float(gamma), _p(idx), _p(do), N, C, d_K,
                                d_V, kk, _p(r) if r is not None else None, nr, _p(dq), _p(dk),
                                _p(dv), _p(dg), int(kind))
    return dq, dk, dv, float(dg[0])


def exact_topk(q, k, C: int, kk: int, rows=None):
    """One slice.  Exact Euclidean top-kk among the prefix keys (float32 inputs)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    kx = np.ascontiguousarray(k, dtype=np.float32)
    N, d_K = q.shape
    r, nr = _rows(rows)
    cnt = nr if r is not None else N
    out = np.empty((cnt, kk), dtype=np.int32)
    _load().orc_exact_topk(_p(q), _p(kx), N, C, d_K, kk, _p(r) if r is not None else None, nr,
                           _p(out))
    return out


# -------------------------------------------------------------- full path ---

def forward(q, k, v, gamma, C: int, k_sel: int, bits: int, rows=None):
    """Whole forward over [B,H,N,.] arrays: encode, select, attend.

    v may be float32/float64 values (bf16 inputs are passed already widened).
    gamma: [H].  rows: optional 1-D query list applied to every slice.
    Returns dict with q_codes, k_codes, idx (int32 [B,H,R,k]), out, rowsum."""
    B, H, N, d_K = q.shape
    qc = encode(q, bits)
    kc = encode(k, bits)
    r, nr = _rows(rows)
    cnt = nr if r is not None else N
    idx = select(qc.reshape(-1, N), kc.reshape(-1, N), C, k_sel, rows=r)
    idx = idx.reshape(B, H, cnt, k_sel)
    out = np.empty((B, H, cnt, v.shape[-1]), dtype=np.float64)
    rs = np.empty((B, H, cnt), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o, s = attend_fwd(q[b, h], k[b, h], v[b, h], float(gamma[h]), idx[b, h], C, rows=r)
            out[b, h] = o
            rs[b, h] = s
    return {"q_codes": qc, "k_codes": kc, "idx": idx, "out": out, "rowsum": rs}
