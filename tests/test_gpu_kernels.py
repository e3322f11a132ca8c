"""GPU parity of the alternative weight kernels (softmax of -|q-k|^2/gamma^2
and inverse Euclidean; OpenReview discussion of "ZETA: Leveraging Z-order
Curves for Efficient Top-k Attention", reply A3 "Justification for Euclidean
Distance Claim").  Selection is the same as for the Cauchy kernel; forward and
backward are compared with the oracle of the same kernel, fed the oracle's own
selection."""
import numpy as np
import pytest
import torch

import oracle
from order_retrieval_gb300 import workloads as W

from gpu_util import Run, assert_close_bf16, assert_close_f32, slice_inputs

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

KIND = {"softmax": oracle.SOFTMAX, "inv_euclid": oracle.INV_EUCLID}


def _check(run, weight, slices, rows=None, backward=True, f32_atol=1e-5):
    w, g = run.w, run.g
    kind = KIND[weight]
    bf16 = w.v_dtype == "bf16"
    close = assert_close_bf16 if bf16 else (
        lambda a, b, what="": assert_close_f32(a, b, atol=f32_atol, what=what))
    idx = run.idx()
    out, rs = run.out(), run.rowsum()
    grads = run.grads() if backward else None
    for s in slices:
        q, k, v, gamma, dout = slice_inputs(w, g, s)
        ref = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None], w.C,
                            w.k, rows=rows)[0]
        assert np.array_equal(idx[s] if rows is None else idx[s][rows], ref)
        o_ref, s_ref = oracle.attend_fwd(q, k, v, gamma, ref, w.C, rows=rows, kind=kind)
        close(out[s] if rows is None else out[s][rows], o_ref, what="out")
        assert_close_f32(rs[s] if rows is None else rs[s][rows], s_ref, what="rowsum")
        if backward:
            dq_r, dk_r, dv_r, _ = oracle.attend_bwd(q, k, v, gamma, ref, dout, w.C, kind=kind)
            close(grads[0][s], dq_r, what="dq")
            close(grads[1][s], dk_r, what="dk")
            close(grads[2][s], dv_r, what="dv")


def _dgamma_ref(run, weight):
    w, g = run.w, run.g
    ref = np.zeros(w.H)
    for s in range(run.S):
        q, k, v, gamma, dout = slice_inputs(w, g, s)
        idx = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None], w.C,
                            w.k)[0]
        ref[s % w.H] += oracle.attend_bwd(q, k, v, gamma, idx, dout, w.C, kind=KIND[weight])[3]
    return ref


@pytest.mark.parametrize("weight", ["softmax", "inv_euclid"])
def test_tiny_f32(weight):
    run = Run(W.TINY, backward=True, weight=weight)
    assert run.status() == 0
    _check(run, weight, (0,))
    dg = run.grads()[3]
    if weight == "inv_euclid":
        assert (dg == 0).all()
    else:
        assert_close_f32(dg, _dgamma_ref(run, weight), what="dgamma")


def test_softmax_small_gamma_needs_the_shift():
    """gamma = 0.05: exp(-d2/gamma^2) alone underflows to 0 for most pairs;
    with the shift the outputs stay finite and match the oracle.  The float32
    rounding of d2 (about 2^-24 d2) enters the weights multiplied by 1/gamma^2,
    so the tolerance is the 1e-5 of gamma = 0.5 scaled by (0.5 / gamma)^2."""
    w = W.TINY.replace(gamma=0.05)
    run = Run(w, backward=True, weight="softmax")
    assert np.isfinite(run.out()).all()
    _check(run, "softmax", (0,), f32_atol=1e-5 * (0.5 / 0.05) ** 2)


@pytest.mark.parametrize("weight", ["softmax", "inv_euclid"])
@pytest.mark.parametrize("d_V", [32, 64])
def test_clustered_bf16(weight, d_V):
    """bf16 values; d_V = 64 takes the tensor-core kernels."""
    w = W.CLUSTERED.replace(B=1, d_V=d_V)
    run = Run(w, backward=True, weight=weight)
    assert run.status() == 0
    _check(run, weight, (0, 5))
    if weight == "softmax":
        assert_close_bf16(run.grads()[3], _dgamma_ref(run, weight), what="dgamma")


TC = [
    dict(N=200, C=40, k=7),
    dict(N=480, C=96, k=33),
    dict(N=256, C=256, k=16),
    dict(N=768, C=192, k=64, d_K=2, bits=12),
    dict(N=512, C=128, k=20, d_K=4, bits=6),
]


@pytest.mark.parametrize("kw", TC, ids=lambda kw: "-".join(f"{a}{b}" for a, b in kw.items()))
@pytest.mark.parametrize("weight", ["softmax", "inv_euclid"])
@pytest.mark.parametrize("gamma", [0.1, (0.3, 1.0)], ids=["g0.1", "g0.3-1"])
def test_tensor_core_shapes(kw, weight, gamma):
    base = dict(name="tck", B=2, H=2, N=256, d_K=3, d_V=64, k=8, C=64, bits=10, v_dtype="bf16",
                gamma=gamma, dist="uniform", v_dist="normal", seed=51)
    base.update(kw)
    w = W.Workload(**base)
    run = Run(w, backward=True, weight=weight)
    assert run.status() == 0
    _check(run, weight, range(run.S))
    if weight == "softmax":
        assert_close_bf16(run.grads()[3], _dgamma_ref(run, weight), what="dgamma")


@pytest.mark.parametrize("weight", ["softmax", "inv_euclid"])
def test_training_workload_sampled(weight):
    """B=4, H=8, N=65536, k=48: forward on sampled rows of two slices,
    backward of one whole slice."""
    run = Run(W.TRAIN, backward=True, weight=weight)
    assert run.status() == 0
    rng = np.random.default_rng(7)
    rows = np.sort(np.concatenate([rng.choice(W.TRAIN.N, 40, replace=False), [0, 1024, 65535]]))
    _check(run, weight, (3,), rows=rows, backward=False)
    _check(run, weight, (17,))
