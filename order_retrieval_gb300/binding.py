"""Thin ctypes binding of libzeta.so with the same names as the C ABI.

Each function only marshals arguments: it checks the torch tensors' dtype,
shape, device and contiguity, then passes raw device pointers and the current
CUDA stream to the library.  Every step of the path runs in the library's CUDA
kernels; there is no fallback of any kind, and a missing library or a failed
build raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

ZETA_F32 = 0
ZETA_BF16 = 1

# Weight kernels (low bits of zeta_problem_t.flags).
ZETA_W_CAUCHY, ZETA_W_SOFTMAX, ZETA_W_INV_EUCLID = 0, 1, 2
WEIGHTS = {"cauchy": ZETA_W_CAUCHY, "softmax": ZETA_W_SOFTMAX, "inv_euclid": ZETA_W_INV_EUCLID}

STATUS = {
    0: "ZETA_OK", 1: "ZETA_ERR_INVALID_ARG", 2: "ZETA_ERR_UNSUPPORTED", 3: "ZETA_ERR_WORKSPACE",
    4: "ZETA_ERR_CUDA", 5: "ZETA_ERR_DEVICE_TIMEOUT", 6: "ZETA_ERR_BOUNDS",
}

HEADER = os.path.join(_build.ROOT, "include", "zeta.h")


class ZetaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class zeta_problem_t(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("d_K", ctypes.c_int32), ("d_V", ctypes.c_int32), ("k", ctypes.c_int32),
                ("C", ctypes.c_int32), ("bits", ctypes.c_int32), ("v_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class zeta_proj_t(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int32), ("F", ctypes.c_int32)]


def problem(B, H, N, d_K, d_V, k, C, bits, v_dtype="bf16", flags=0,
            weight="cauchy") -> zeta_problem_t:
    """flags: raw flag bits; weight: 'cauchy', 'softmax' or 'inv_euclid' (ORed in)."""
    vd = {"f32": ZETA_F32, "bf16": ZETA_BF16, ZETA_F32: ZETA_F32, ZETA_BF16: ZETA_BF16}[v_dtype]
    return zeta_problem_t(B, H, N, d_K, d_V, k, C, bits, vd, flags | WEIGHTS[weight])


def problem_of(w, weight="cauchy") -> zeta_problem_t:
    """Problem struct of a workloads.Workload."""
    return problem(w.B, w.H, w.N, w.d_K, w.d_V, w.k, w.C, w.bits, w.v_dtype, weight=weight)


_lib = None


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libzeta.so (building it in-tree first if needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"ZETA CUDA library not found at {path}")
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    PP = ctypes.POINTER(zeta_problem_t)
    S = ctypes.c_int
    L.zeta_code_bytes.argtypes = [PP]
    L.zeta_code_bytes.restype = ctypes.c_size_t
    L.zeta_prefix_entries.argtypes = [PP]
    L.zeta_prefix_entries.restype = ctypes.c_int64
    L.zeta_sort_workspace_bytes.argtypes = [PP]
    L.zeta_sort_workspace_bytes.restype = ctypes.c_size_t
    L.zeta_bwd_workspace_bytes.argtypes = [PP]
    L.zeta_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.zeta_status_string.argtypes = [S]
    L.zeta_status_string.restype = ctypes.c_char_p
    L.zeta_encode.argtypes = [PP, P, P, P]
    L.zeta_encode.restype = S
    L.zeta_sort_chunks.argtypes = [PP, P, P, P, P, ctypes.c_size_t, P]
    L.zeta_sort_chunks.restype = S
    L.zeta_select_topk.argtypes = [PP, P, P, P, P, P]
    L.zeta_select_topk.restype = S
    L.zeta_encode_curves.argtypes = [PP, P, ctypes.c_int32, P, P, P]
    L.zeta_encode_curves.restype = S
    L.zeta_select_topk_curves.argtypes = [PP, ctypes.c_int32, P, P, P, P, P]
    L.zeta_select_topk_curves.restype = S
    L.zeta_project_encode.argtypes = [PP, ctypes.POINTER(zeta_proj_t)] + [P] * 11
    L.zeta_project_encode.restype = S
    L.zeta_attend_fwd.argtypes = [PP, P, P, P, P, P, P, P, P, P]
    L.zeta_attend_fwd.restype = S
    L.zeta_attend_bwd.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    L.zeta_select_attend_fwd.argtypes = [PP] + [P] * 12
    L.zeta_check_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.c_int32, P, P]
    L.zeta_check_bounded_wait.restype = S
    L.zeta_select_attend_fwd.restype = S
    L.zeta_attend_bwd.restype = S
    _lib = L
    return L


def header_functions() -> list:
    """Names of the functions declared in include/zeta.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zeta_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------- marshalling ---

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("ZETA tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("ZETA tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code):
    if code != 0:
        raise ZetaError(fn, code)


def _expect(t, name, dtype, numel):
    if t is None:
        return
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")


def code_dtype(p: zeta_problem_t):
    return torch.int64 if p.d_K * p.bits > 32 else torch.int32


def v_torch_dtype(p: zeta_problem_t):
    return torch.bfloat16 if p.v_dtype == ZETA_BF16 else torch.float32


def zeta_code_bytes(p: zeta_problem_t) -> int:
    return lib().zeta_code_bytes(ctypes.byref(p))


def zeta_prefix_entries(p: zeta_problem_t) -> int:
    return lib().zeta_prefix_entries(ctypes.byref(p))


def zeta_sort_workspace_bytes(p: zeta_problem_t) -> int:
    return lib().zeta_sort_workspace_bytes(ctypes.byref(p))


def zeta_bwd_workspace_bytes(p: zeta_problem_t) -> int:
    return lib().zeta_bwd_workspace_bytes(ctypes.byref(p))


def zeta_status_string(code: int) -> str:
    return lib().zeta_status_string(code).decode()


def zeta_encode(p, x, codes, stream=None):
    S = p.B * p.H * p.N
    _expect(x, "x", torch.float32, S * p.d_K)
    _expect(codes, "codes", code_dtype(p), S)
    _check("zeta_encode", lib().zeta_encode(ctypes.byref(p), _ptr(x), _ptr(codes), _stream(stream)))


def zeta_sort_chunks(p, key_codes, prefix_codes, prefix_idx, workspace, stream=None):
    S = p.B * p.H
    T = zeta_prefix_entries(p)
    _expect(key_codes, "key_codes", code_dtype(p), S * p.N)
    _expect(prefix_codes, "prefix_codes", code_dtype(p), S * T)
    _expect(prefix_idx, "prefix_idx", torch.int32, S * T)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("zeta_sort_chunks",
           lib().zeta_sort_chunks(ctypes.byref(p), _ptr(key_codes), _ptr(prefix_codes),
                                  _ptr(prefix_idx), _ptr(workspace), ws_bytes, _stream(stream)))


def zeta_sort_chunks_noalloc(p, key_codes, prefix_codes, prefix_idx, stream=None):
    """zeta_sort_chunks with the library's own fixed 32 MiB device scratch
    (for callers that cannot allocate a workspace)."""
    L = lib()
    fn = L.zeta_sort_chunks_noalloc
    fn.argtypes = [ctypes.POINTER(zeta_problem_t), ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    S = p.B * p.H
    T = zeta_prefix_entries(p)
    _expect(key_codes, "key_codes", code_dtype(p), S * p.N)
    _expect(prefix_codes, "prefix_codes", code_dtype(p), S * T)
    _expect(prefix_idx, "prefix_idx", torch.int32, S * T)
    _check("zeta_sort_chunks_noalloc",
           fn(ctypes.byref(p), _ptr(key_codes), _ptr(prefix_codes), _ptr(prefix_idx),
              _stream(stream)))


def zeta_select_topk(p, q_codes, prefix_codes, prefix_idx, idx, stream=None):
    S = p.B * p.H
    _expect(q_codes, "q_codes", code_dtype(p), S * p.N)
    _expect(idx, "idx", torch.int32, S * p.N * p.k)
    _check("zeta_select_topk",
           lib().zeta_select_topk(ctypes.byref(p), _ptr(q_codes), _ptr(prefix_codes),
                                  _ptr(prefix_idx), _ptr(idx), _stream(stream)))


def zeta_encode_curves(p, x, axes, codes, stream=None):
    """axes: sequence of `curves` coordinate orders (each a permutation of
    0..d_K-1); codes: [curves * B * H * N] of the problem's code type."""
    rows = [list(map(int, a)) for a in axes]
    curves = len(rows)
    S = p.B * p.H * p.N
    _expect(x, "x", torch.float32, S * p.d_K)
    _expect(codes, "codes", code_dtype(p), curves * S)
    flat = [v for r in rows for v in r]
    if any(len(r) != p.d_K for r in rows):
        raise ValueError("every axis order needs d_K entries")
    arr = (ctypes.c_int32 * max(1, len(flat)))(*flat)
    _check("zeta_encode_curves",
           lib().zeta_encode_curves(ctypes.byref(p), _ptr(x), curves, arr, _ptr(codes),
                                    _stream(stream)))


def zeta_select_topk_curves(p, curves, q_codes, prefix_codes, prefix_idx, idx, stream=None):
    S = p.B * p.H
    T = zeta_prefix_entries(p)
    _expect(q_codes, "q_codes", code_dtype(p), curves * S * p.N)
    _expect(prefix_codes, "prefix_codes", code_dtype(p), curves * S * T)
    _expect(prefix_idx, "prefix_idx", torch.int32, curves * S * T)
    _expect(idx, "idx", torch.int32, S * p.N * p.k)
    _check("zeta_select_topk_curves",
           lib().zeta_select_topk_curves(ctypes.byref(p), curves, _ptr(q_codes),
                                         _ptr(prefix_codes), _ptr(prefix_idx), _ptr(idx),
                                         _stream(stream)))


def zeta_project_encode(p, D, F, x, w1, b1, w2, b2, q, k, q_codes, k_codes, dev_status=None,
                        stream=None):
    """x bf16 [B,N,D]; w1 bf16 [2,H*F,D]; b1 f32 [2,H*F]; w2 f32 [2,H,d_K,F];
    b2 f32 [2,H,d_K]; q, k f32 [B,H,N,d_K]; q_codes, k_codes [B,H,N]."""
    S = p.B * p.H * p.N
    _expect(x, "x", torch.bfloat16, p.B * p.N * D)
    _expect(w1, "w1", torch.bfloat16, 2 * p.H * F * D)
    _expect(b1, "b1", torch.float32, 2 * p.H * F)
    _expect(w2, "w2", torch.float32, 2 * p.H * p.d_K * F)
    _expect(b2, "b2", torch.float32, 2 * p.H * p.d_K)
    for t, n in ((q, "q"), (k, "k")):
        _expect(t, n, torch.float32, S * p.d_K)
    for t, n in ((q_codes, "q_codes"), (k_codes, "k_codes")):
        _expect(t, n, code_dtype(p), S)
    _expect(dev_status, "dev_status", torch.int32, 1)
    pj = zeta_proj_t(D, F)
    _check("zeta_project_encode",
           lib().zeta_project_encode(ctypes.byref(p), ctypes.byref(pj), _ptr(x), _ptr(w1),
                                     _ptr(b1), _ptr(w2), _ptr(b2), _ptr(q), _ptr(k),
                                     _ptr(q_codes), _ptr(k_codes), _ptr(dev_status),
                                     _stream(stream)))


def zeta_check_bounded_wait(iterations, arrive, dev_status, stream=None):
    """Run the kernels' bounded mbarrier wait on a barrier that is (arrive=1) or
    is not (arrive=0) completed; a wait that gives up writes
    ZETA_ERR_DEVICE_TIMEOUT to dev_status."""
    _expect(dev_status, "dev_status", torch.int32, 1)
    _check("zeta_check_bounded_wait",
           lib().zeta_check_bounded_wait(int(iterations), int(arrive), _ptr(dev_status),
                                         _stream(stream)))


def curve_axes(d_K: int, curves: int) -> list:
    """The pages' coordinate orders: one curve = (0..d_K-1); three = the cyclic
    shifts of (0, 1, 2); six = all orderings of (0, 1, 2)."""
    if curves == 1:
        return [list(range(d_K))]
    if d_K != 3:
        raise ValueError("several curves are defined for d_K = 3")
    if curves == 3:
        return [[0, 1, 2], [1, 2, 0], [2, 0, 1]]
    if curves == 6:
        return [[0, 1, 2], [0, 2, 1], [1, 2, 0], [1, 0, 2], [2, 0, 1], [2, 1, 0]]
    raise ValueError("curves must be 1, 3 or 6")


def zeta_attend_fwd(p, q, k, v, gamma, idx, out, rowsum, dev_status=None, stream=None):
    S = p.B * p.H * p.N
    vt = v_torch_dtype(p)
    _expect(q, "q", torch.float32, S * p.d_K)
    _expect(k, "k", torch.float32, S * p.d_K)
    _expect(v, "v", vt, S * p.d_V)
    _expect(gamma, "gamma", torch.float32, p.H)
    _expect(idx, "idx", torch.int32, S * p.k)
    _expect(out, "out", vt, S * p.d_V)
    _expect(rowsum, "rowsum", torch.float32, S)
    _expect(dev_status, "dev_status", torch.int32, 1)
    _check("zeta_attend_fwd",
           lib().zeta_attend_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                 _ptr(idx), _ptr(out), _ptr(rowsum), _ptr(dev_status),
                                 _stream(stream)))


def zeta_select_attend_fwd(p, q, k, v, gamma, q_codes, prefix_codes, prefix_idx, idx, out,
                           rowsum, dev_status=None, stream=None):
    S = p.B * p.H * p.N
    vt = v_torch_dtype(p)
    T = zeta_prefix_entries(p)
    _expect(q, "q", torch.float32, S * p.d_K)
    _expect(k, "k", torch.float32, S * p.d_K)
    _expect(v, "v", vt, S * p.d_V)
    _expect(gamma, "gamma", torch.float32, p.H)
    _expect(q_codes, "q_codes", code_dtype(p), S)
    _expect(prefix_codes, "prefix_codes", code_dtype(p), p.B * p.H * T)
    _expect(prefix_idx, "prefix_idx", torch.int32, p.B * p.H * T)
    _expect(idx, "idx", torch.int32, S * p.k)
    _expect(out, "out", vt, S * p.d_V)
    _expect(rowsum, "rowsum", torch.float32, S)
    _expect(dev_status, "dev_status", torch.int32, 1)
    _check("zeta_select_attend_fwd",
           lib().zeta_select_attend_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                        _ptr(q_codes), _ptr(prefix_codes), _ptr(prefix_idx),
                                        _ptr(idx), _ptr(out), _ptr(rowsum), _ptr(dev_status),
                                        _stream(stream)))


def zeta_attend_bwd(p, q, k, v, gamma, idx, dout, dq, dk, dv, dgamma, workspace,
                    dev_status=None, stream=None):
    S = p.B * p.H * p.N
    vt = v_torch_dtype(p)
    _expect(q, "q", torch.float32, S * p.d_K)
    _expect(k, "k", torch.float32, S * p.d_K)
    _expect(v, "v", vt, S * p.d_V)
    _expect(gamma, "gamma", torch.float32, p.H)
    _expect(idx, "idx", torch.int32, S * p.k)
    _expect(dout, "dout", vt, S * p.d_V)
    _expect(dq, "dq", torch.float32, S * p.d_K)
    _expect(dk, "dk", torch.float32, S * p.d_K)
    _expect(dv, "dv", vt, S * p.d_V)
    _expect(dgamma, "dgamma", torch.float32, p.H)
    _expect(dev_status, "dev_status", torch.int32, 1)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("zeta_attend_bwd",
           lib().zeta_attend_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                 _ptr(idx), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(dgamma), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                 _stream(stream)))
