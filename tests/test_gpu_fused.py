"""GPU parity of the fused select + attend call (zeta_select_attend_fwd).

The window indices it writes must equal the oracle's selection bit for bit, and
its outputs must equal those of zeta_select_topk followed by zeta_attend_fwd
bit for bit (the same arithmetic on the same windows); one slice per case is
also checked against the oracle's forward."""
import numpy as np
import pytest
import torch

import oracle
from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W
from order_retrieval_gb300.pipeline import ZetaPlan

from gpu_util import (assert_close_bf16, assert_close_f32, dev_vals, host_vals, in_threads,
                      slice_inputs)

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def _run(w, weight="cauchy", rows=None, slices=(0,), full=()):
    """Fused and two-call forwards of w, bit for bit equal; the listed slices
    against the oracle on `rows` (all rows when None), the slices in `full` on
    all rows."""
    g = W.generate(w)
    p = zb.problem_of(w, weight=weight)
    q = torch.from_numpy(g["q"]).cuda().reshape(-1)
    k = torch.from_numpy(g["k"]).cuda().reshape(-1)
    v = dev_vals(w, g["v"]).reshape(-1)
    gm = torch.from_numpy(g["gamma"]).cuda()
    two = ZetaPlan(p, "cuda", backward=False)
    one = ZetaPlan(p, "cuda", backward=False, fused=True)
    one.idx.fill_(12345)                      # every entry must be written
    two.forward(q, k, v, gm)
    one.forward(q, k, v, gm)
    torch.cuda.synchronize()
    assert int(one.status.item()) == 0 and int(two.status.item()) == 0
    assert torch.equal(one.idx, two.idx)
    assert torch.equal(one.out, two.out)
    assert torch.equal(one.rowsum, two.rowsum)
    S = w.B * w.H
    idx = one.idx.cpu().numpy().reshape(S, w.N, w.k)
    out = host_vals(one.out).reshape(S, w.N, w.d_V)
    rs = one.rowsum.cpu().numpy().astype(np.float64).reshape(S, w.N)
    kind = {"cauchy": oracle.CAUCHY, "softmax": oracle.SOFTMAX, "inv_euclid": oracle.INV_EUCLID}

    def check(case):
        s, r = case
        qs, ks, vs, gamma, _ = slice_inputs(w, g, s)
        ref = oracle.select(oracle.encode(qs, w.bits)[None], oracle.encode(ks, w.bits)[None],
                            w.C, w.k, rows=r)[0]
        sel = slice(None) if r is None else r
        assert np.array_equal(idx[s][sel], ref)
        o_ref, s_ref = oracle.attend_fwd(qs, ks, vs, gamma, ref, w.C, rows=r,
                                         kind=kind[weight])
        close = assert_close_bf16 if w.v_dtype == "bf16" else assert_close_f32
        close(out[s][sel], o_ref, what="out")
        assert_close_f32(rs[s][sel], s_ref, what="rowsum")

    in_threads(check, [(s, rows) for s in slices] + [(s, None) for s in full])


def test_tiny_f32_takes_the_two_call_path():
    _run(W.TINY)


@pytest.mark.parametrize("weight", ["cauchy", "softmax", "inv_euclid"])
def test_clustered_bf16(weight):
    _run(W.CLUSTERED.replace(B=1), weight=weight, slices=(0, 7))


@pytest.mark.parametrize("kw", [dict(N=200, C=40, k=7), dict(N=256, C=256, k=16),
                                dict(N=480, C=96, k=33), dict(N=512, C=64, k=64, bits=1),
                                dict(N=768, C=192, k=64, d_K=2, bits=12),
                                dict(N=512, C=128, k=20, d_K=4, bits=6)],
                         ids=lambda kw: "-".join(f"{a}{b}" for a, b in kw.items()))
def test_tensor_core_shapes(kw):
    base = dict(name="fused", B=2, H=2, N=256, d_K=3, d_V=64, k=8, C=64, bits=10, v_dtype="bf16",
                gamma=(0.3, 1.0), dist="uniform", v_dist="normal", seed=61)
    base.update(kw)
    _run(W.Workload(**base), slices=(0, 3))


@pytest.mark.parametrize("w", [W.EFFICIENCY, W.PAGES12], ids=lambda w: w.name)
def test_efficiency_scale_full_slice(w):
    """The timed 65,536-token workload (and the pages' 12-bit grid): every
    slice of the fused call equal to the two-call path bit for bit, slice 5
    whole against the oracle element by element, slice 0 on sampled rows."""
    rng = np.random.default_rng(5)
    rows = np.sort(np.concatenate([rng.choice(w.N, 40, replace=False), [0, w.C, w.N - 1]]))
    _run(w, rows=rows, slices=(0,), full=(5,))


@pytest.mark.parametrize("kw", [dict(N=262144, C=1024, bits=12), dict(N=524288, C=2048, bits=10)],
                         ids=["n262144-u64", "n524288-u32"])
def test_long_prefixes(kw):
    """Prefixes long enough that the fused call's first-level table holds the
    first code of every 128 or more entries (64-bit codes at N = 262,144,
    32-bit codes at N = 524,288): every row equal to the two-call path, rows of
    three chunks against the oracle."""
    w = W.EFFICIENCY.replace(name="fused_long", H=1, k=64, **kw)
    n = w.N // w.C
    rows = np.concatenate([np.arange(c * w.C, c * w.C + 24) for c in (1, n // 2, n - 1)])
    _run(w, rows=rows, slices=(0,))
