"""Host-side checks of the C-ABI library: it builds, loads without a GPU,
exports every function include/zeta.h declares, and rejects invalid requests
before launching anything (these calls never reach the CUDA runtime)."""
import ctypes
import subprocess

import pytest

from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import build as zbuild
from order_retrieval_gb300 import workloads as W


@pytest.fixture(scope="module")
def L():
    return zb.lib()


def test_library_exports_every_header_function(L):
    names = zb.header_functions()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", zbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)
    # Only the ABI is exported: internal launchers stay hidden.
    assert not [e for e in exported if "launch_" in e]


def test_status_strings(L):
    for code, name in zb.STATUS.items():
        assert zb.zeta_status_string(code) == name


def test_sizes_follow_the_problem():
    for w in (W.TINY, W.CLUSTERED, W.EFFICIENCY, W.LONG, W.TRAIN, *W.SWEEP):
        p = zb.problem_of(w)
        assert zb.zeta_prefix_entries(p) == w.prefix_entries
        assert zb.zeta_code_bytes(p) == (8 if w.d_K * w.bits > 32 else 4)
        assert zb.zeta_sort_workspace_bytes(p) > 0
        assert zb.zeta_bwd_workspace_bytes(p) > 0
    p = zb.problem_of(W.EFFICIENCY)
    assert zb.zeta_prefix_entries(p) == 1024 * 64 * 63 // 2


BAD = [
    dict(N=1000),                 # C does not divide N
    dict(k=0), dict(k=2000),      # k outside [1, C]
    dict(d_K=0), dict(bits=0), dict(C=0), dict(d_V=0),
    dict(d_K=8, bits=9),          # 72-bit code
    dict(B=-1), dict(v_dtype=7),
]
UNSUP = [dict(d_K=9, bits=7), dict(bits=25, d_K=2), dict(d_V=512), dict(flags=3),
         dict(flags=4)]


def _prob(**kw):
    base = dict(B=1, H=2, N=1024, d_K=3, d_V=32, k=16, C=128, bits=10, v_dtype="f32")
    base.update(kw)
    flags = base.pop("flags", 0)
    vd = base.pop("v_dtype")
    p = zb.problem(**base, v_dtype="f32" if vd not in (0, 1, "f32", "bf16") else vd, flags=flags)
    if vd not in (0, 1, "f32", "bf16"):
        p.v_dtype = vd
    return p


@pytest.mark.parametrize("kw", BAD)
def test_invalid_problems_are_rejected_without_launch(L, kw):
    p = _prob(**kw)
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the checks fail first
    assert L.zeta_encode(P, fake, fake, None) == 1
    assert L.zeta_select_topk(P, fake, fake, fake, fake, None) == 1
    assert L.zeta_attend_fwd(P, fake, fake, fake, fake, fake, fake, fake, None, None) == 1
    assert L.zeta_prefix_entries(P) == -1
    assert L.zeta_code_bytes(P) == 0
    assert L.zeta_sort_workspace_bytes(P) == 0


@pytest.mark.parametrize("kw", UNSUP)
def test_unsupported_problems(L, kw):
    p = _prob(**kw)
    fake = ctypes.c_void_p(0x1000)
    assert L.zeta_encode(ctypes.byref(p), fake, fake, None) == 2


def test_null_pointers_and_workspace(L):
    p = _prob()
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x1000)
    assert L.zeta_encode(None, fake, fake, None) == 1
    assert L.zeta_encode(P, None, fake, None) == 1
    assert L.zeta_select_topk(P, fake, fake, fake, None, None) == 1
    ws = zb.zeta_sort_workspace_bytes(p)
    assert L.zeta_sort_chunks(P, fake, fake, fake, None, ws, None) == 3
    assert L.zeta_sort_chunks(P, fake, fake, fake, ctypes.c_void_p(0x10000), ws - 1, None) == 3
    assert L.zeta_sort_chunks(P, fake, fake, fake, ctypes.c_void_p(0x10010), ws, None) == 3
    bws = zb.zeta_bwd_workspace_bytes(p)
    args = [fake] * 10
    assert L.zeta_attend_bwd(P, *args, None, bws, None, None) == 3
    assert L.zeta_attend_bwd(P, *args, ctypes.c_void_p(0x10000), bws - 1, None, None) == 3
    assert L.zeta_attend_bwd(P, *args, ctypes.c_void_p(0x10010), bws, None, None) == 3
    # Unaligned value pointers are refused.
    odd = ctypes.c_void_p(0x1002)
    assert L.zeta_attend_fwd(P, fake, fake, odd, fake, fake, fake, fake, None, None) == 1
    # Too many chunks for the prefix builder.
    many = _prob(N=4096, C=2, k=2)
    assert L.zeta_sort_chunks(ctypes.byref(many), fake, fake, fake, fake, 1 << 40, None) == 2


def test_weight_kernels_are_accepted(L):
    for wk in ("cauchy", "softmax", "inv_euclid"):
        p = zb.problem(1, 2, 1024, 3, 32, 16, 128, 10, "f32", weight=wk)
        assert L.zeta_prefix_entries(ctypes.byref(p)) > 0
        assert zb.zeta_bwd_workspace_bytes(p) > 0


def test_empty_problems_are_no_ops(L):
    for kw in (dict(B=0), dict(N=0), dict(H=0)):
        p = _prob(**kw)
        P = ctypes.byref(p)
        assert L.zeta_encode(P, None, None, None) == 0
        assert L.zeta_select_topk(P, None, None, None, None, None) == 0
        assert L.zeta_attend_fwd(P, None, None, None, None, None, None, None, None, None) == 0


def test_curve_calls_check_their_arguments(L):
    p = _prob(k=16)
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x1000)
    Ax = ctypes.c_int32 * 24

    def enc(curves, rows):
        flat = [v for r in rows for v in r]
        return L.zeta_encode_curves(P, fake, curves, Ax(*flat), fake, None)

    assert enc(0, []) == 1                                      # no curve
    assert enc(9, [[0, 1, 2]] * 8) == 1                         # above 8 curves
    assert enc(2, [[0, 1, 2], [0, 0, 2]]) == 1                  # repeated axis
    assert enc(1, [[0, 1, 3]]) == 1                             # axis out of range
    assert L.zeta_encode_curves(P, fake, 3, None, fake, None) == 1
    assert L.zeta_encode_curves(P, None, 1, Ax(0, 1, 2), fake, None) == 1
    assert L.zeta_select_topk_curves(P, 0, fake, fake, fake, fake, None) == 1
    assert L.zeta_select_topk_curves(P, 17, fake, fake, fake, fake, None) == 1  # k // 17 == 0
    assert L.zeta_select_topk_curves(P, 3, fake, fake, fake, None, None) == 1
    big = _prob(k=512, C=512)
    assert L.zeta_select_topk_curves(ctypes.byref(big), 3, fake, fake, fake, fake, None) == 2
    for kw in (dict(B=0), dict(N=0)):
        e = _prob(**kw)
        assert L.zeta_encode_curves(ctypes.byref(e), None, 3, Ax(0, 1, 2, 1, 2, 0, 2, 0, 1),
                                    None, None) == 0
        assert L.zeta_select_topk_curves(ctypes.byref(e), 3, None, None, None, None, None) == 0
    assert zb.curve_axes(3, 6)[3] == [1, 0, 2]


def test_project_encode_checks_its_arguments(L):
    p = _prob(H=8)
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x1000)
    ok = zb.zeta_proj_t(512, 64)
    args = [fake] * 11
    assert L.zeta_project_encode(P, None, *args) == 1                        # no widths
    assert L.zeta_project_encode(P, ctypes.byref(zb.zeta_proj_t(0, 64)), *args) == 1
    assert L.zeta_project_encode(P, ctypes.byref(ok), None, *args[1:]) == 1  # null x
    odd = [ctypes.c_void_p(0x1008)] + args[1:]
    assert L.zeta_project_encode(P, ctypes.byref(ok), *odd) == 1             # x not 16-B aligned
    for pj in (zb.zeta_proj_t(512, 32), zb.zeta_proj_t(500, 64)):             # F != 64, D % 64
        assert L.zeta_project_encode(P, ctypes.byref(pj), *args) == 2
    p6 = _prob(H=6)
    assert L.zeta_project_encode(ctypes.byref(p6), ctypes.byref(ok), *args) == 2   # H % 4
    e = _prob(B=0)
    assert L.zeta_project_encode(ctypes.byref(e), ctypes.byref(ok), *([None] * 11)) == 0
    # the binding's marshalling matches the C signature (empty problem: no launch)
    pe = zb.problem(0, 8, 1024, 3, 64, 16, 128, 10, "bf16")
    zb.zeta_project_encode(pe, 512, 64, *([None] * 9), stream=0)


def test_select_attend_checks_its_arguments(L):
    p = _prob()
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x1000)
    args = [fake] * 12
    assert L.zeta_select_attend_fwd(None, *args) == 1
    for pos in (0, 1, 2, 3, 4, 7, 8, 9):          # q, k, v, gamma, q_codes, idx, out, rowsum
        bad = list(args)
        bad[pos] = None
        assert L.zeta_select_attend_fwd(P, *bad) == 1, pos
    odd = list(args)
    odd[2] = ctypes.c_void_p(0x1002)               # v not 16-B aligned
    assert L.zeta_select_attend_fwd(P, *odd) == 1
    assert L.zeta_select_attend_fwd(ctypes.byref(_prob(N=1000)), *args) == 1
    e = _prob(B=0)
    assert L.zeta_select_attend_fwd(ctypes.byref(e), *([None] * 12)) == 0
    pe = zb.problem(0, 2, 1024, 3, 32, 16, 128, 10, "f32")
    zb.zeta_select_attend_fwd(pe, *([None] * 10), stream=0)


def test_bounded_wait_check_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    assert L.zeta_check_bounded_wait(100, 0, None, None) == 1
    assert L.zeta_check_bounded_wait(0, 0, fake, None) == 1
