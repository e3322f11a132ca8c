"""GPU parity of the multi-curve variant (three cyclic or six permuted
coordinate orders, k // curves window keys per curve, union of the windows).

Codes and selected rows are bit-exact against the oracle; forward and backward
results against the oracle within the bf16 / fp32 criteria, fed with the
oracle's own selection.
"""
import numpy as np
import pytest
import torch

import oracle
from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W
from order_retrieval_gb300.pipeline import ZetaPlan

from gpu_util import assert_close_bf16, assert_close_f32, codes_np, dev_vals, host_vals, slice_inputs

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


class CurveRun:
    def __init__(self, w, curves, backward=False):
        self.w, self.curves = w, curves
        self.g = W.generate(w, with_dout=backward)
        self.p = zb.problem_of(w)
        self.S = w.B * w.H
        self.q = torch.from_numpy(self.g["q"]).cuda().reshape(-1)
        self.k = torch.from_numpy(self.g["k"]).cuda().reshape(-1)
        self.v = dev_vals(w, self.g["v"]).reshape(-1)
        self.gamma = torch.from_numpy(self.g["gamma"]).cuda()
        self.plan = ZetaPlan(self.p, "cuda", backward=backward, curves=curves)
        self.plan.forward(self.q, self.k, self.v, self.gamma)
        if backward:
            self.dout = dev_vals(w, self.g["dout"]).reshape(-1)
            self.plan.backward(self.q, self.k, self.v, self.gamma, self.dout)
        torch.cuda.synchronize()
        assert int(self.plan.status.item()) == 0

    def idx(self):
        return self.plan.idx.cpu().numpy().reshape(self.S, self.w.N, self.w.k)


def _check(run, slices, rows=None, backward=False):
    w = run.w
    bf16 = w.v_dtype == "bf16"
    close = assert_close_bf16 if bf16 else assert_close_f32
    idx = run.idx()
    out = host_vals(run.plan.out).reshape(run.S, w.N, w.d_V)
    rs = run.plan.rowsum.cpu().numpy().astype(np.float64).reshape(run.S, w.N)
    for s in slices:
        q, k, v, gamma, dout = slice_inputs(w, run.g, s)
        ref = oracle.select_multi(q, k, w.C, w.k, w.bits, run.curves, rows=rows)
        got = idx[s] if rows is None else idx[s][rows]
        assert np.array_equal(got, ref)
        o_ref, s_ref = oracle.attend_fwd(q, k, v, gamma, ref, w.C, rows=rows)
        close(out[s] if rows is None else out[s][rows], o_ref, what="out")
        assert_close_f32(rs[s] if rows is None else rs[s][rows], s_ref, what="rowsum")
        if backward:
            dq_r, dk_r, dv_r, _ = oracle.attend_bwd(q, k, v, gamma, ref, dout, w.C)
            dq = run.plan.dq.cpu().numpy().astype(np.float64).reshape(run.S, w.N, w.d_K)
            dk = run.plan.dk.cpu().numpy().astype(np.float64).reshape(run.S, w.N, w.d_K)
            dv = host_vals(run.plan.dv).reshape(run.S, w.N, w.d_V)
            close(dq[s], dq_r, what="dq")
            close(dk[s], dk_r, what="dk")
            close(dv[s], dv_r, what="dv")


@pytest.mark.parametrize("curves", [3, 6])
@pytest.mark.parametrize("bits", [10, 12])
def test_encode_curves_bit_exact(curves, bits):
    w = W.CLUSTERED.replace(B=1, H=2, bits=bits)
    g = W.generate(w)
    p = zb.problem_of(w)
    x = torch.from_numpy(g["q"]).cuda().reshape(-1)
    axes = zb.curve_axes(3, curves)
    codes = torch.empty(curves * w.H * w.N, dtype=zb.code_dtype(p), device="cuda")
    zb.zeta_encode_curves(p, x, axes, codes)
    got = codes_np(codes).reshape(curves, w.H * w.N)
    for m, a in enumerate(axes):
        assert np.array_equal(got[m], oracle.encode_axes(g["q"], bits, a).reshape(-1))


@pytest.mark.parametrize("d_K,bits", [(2, 20), (5, 6)])
def test_encode_curves_other_widths(d_K, bits):
    """Any permutation of any d_K: the general bit-loop path."""
    w = W.TINY.replace(d_K=d_K, bits=bits)
    g = W.generate(w)
    p = zb.problem_of(w)
    x = torch.from_numpy(g["q"]).cuda().reshape(-1)
    rng = np.random.default_rng(d_K)
    axes = [list(range(d_K))] + [rng.permutation(d_K).tolist() for _ in range(3)]
    codes = torch.empty(4 * w.N, dtype=zb.code_dtype(p), device="cuda")
    zb.zeta_encode_curves(p, x, axes, codes)
    got = codes_np(codes).reshape(4, w.N)
    for m, a in enumerate(axes):
        assert np.array_equal(got[m], oracle.encode_axes(g["q"][0, 0], bits, a))


@pytest.mark.parametrize("curves", [3, 6])
def test_clustered_forward_and_backward(curves):
    """The clustered workload (N=4096, C=256, k=32, per-head gamma): k=32 gives
    10 (3 curves) or 5 (6 curves) keys per curve, so rows end in padding."""
    run = CurveRun(W.CLUSTERED.replace(B=1), curves, backward=True)
    _check(run, (0, 5), backward=True)


@pytest.mark.parametrize("kw", [dict(k=100, C=128), dict(k=64, C=64, bits=12),
                                dict(k=7, C=32, bits=2)],
                         ids=["k100-4blocks", "k64-u64codes", "k7-heavy-ties"])
@pytest.mark.parametrize("curves", [3, 6])
def test_small_shapes(kw, curves):
    base = dict(name="curves", B=1, H=2, N=512, d_K=3, d_V=16, k=16, C=64, bits=10,
                v_dtype="f32", gamma=(0.3, 1.0), dist="uniform", v_dist="normal", seed=41)
    base.update(kw)
    w = W.Workload(**base)
    run = CurveRun(w, curves, backward=True)
    _check(run, range(run.S), backward=True)


def test_one_curve_plan_is_the_single_curve_path():
    w = W.CLUSTERED.replace(B=1, H=2)
    run = CurveRun(w, 1)
    q, k, _, _, _ = slice_inputs(w, run.g, 1)
    ref = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None], w.C,
                        w.k)[0]
    assert np.array_equal(run.idx()[1], ref)


@pytest.mark.parametrize("curves", [3, 6])
def test_efficiency_scale_sampled(curves):
    """N = 65536, C = 1024, k = 64 (the efficiency workload) on sampled rows."""
    w = W.EFFICIENCY
    run = CurveRun(w, curves)
    rng = np.random.default_rng(curves)
    rows = np.sort(np.concatenate([rng.choice(w.N, 24, replace=False),
                                   [0, w.C - 1, w.C, w.N - 1]]))
    _check(run, (0, 7), rows=rows)
