"""GPU parity on the long-sequence workload (N = 1,048,576, C = 4096, k = 64,
bf16 values) and the locality side sweep (N = 16384, d_K in {1, 2, 3, 8}).

At N = 1M the prefix table has 1.07 G entries, so it is checked on the device
by properties that pin it completely (each prefix sorted by (code, index) and
holding exactly the indices 0..cC-1) plus exact comparisons of three prefixes;
selected indices and outputs are compared with the oracle on sampled queries.
The sweep also measures how many of the exact Euclidean top-k neighbours the
Z-order window keeps (recall)."""
import numpy as np
import pytest
import torch

import oracle
from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W

from gpu_util import Run, assert_close_bf16, assert_close_f32, codes_np, slice_inputs

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def _prefix_properties_on_device(pc, pi, w, S):
    """Every prefix c: codes non-decreasing, equal codes in increasing index
    order, and the indices are exactly 0..cC-1 (checked through their count,
    sum and sum of squares together with the ordering)."""
    T = w.prefix_entries
    C, n = w.C, w.n_chunks
    pc = pc.view(S, T).to(torch.int64) & 0xFFFFFFFF if pc.dtype == torch.int32 else pc.view(S, T)
    pi = pi.view(S, T).to(torch.int64)
    for c in range(1, n):
        off = C * c * (c - 1) // 2
        M = c * C
        code = pc[:, off:off + M]
        ix = pi[:, off:off + M]
        dc = code[:, 1:] - code[:, :-1]
        assert bool((dc >= 0).all())
        tie = dc == 0
        assert bool(((ix[:, 1:] - ix[:, :-1])[tie] > 0).all())
        assert bool(((ix >= 0) & (ix < M)).all())
        assert bool((ix.sum(1) == M * (M - 1) // 2).all())
        sq = (ix * ix).sum(1)
        assert bool((sq == (M - 1) * M * (2 * M - 1) // 6).all())


def test_long_sequence_forward_sampled():
    w = W.LONG
    run = Run(w)
    assert run.status() == 0
    g = run.g
    S = run.S
    for name, got in (("q", run.q_codes()), ("k", run.k_codes())):
        assert np.array_equal(got, oracle.encode(g[name], w.bits).reshape(S, w.N))
    _prefix_properties_on_device(run.plan.prefix_codes, run.plan.prefix_idx, w, S)
    kc = oracle.encode(g["k"], w.bits).reshape(S, w.N)
    T = w.prefix_entries
    for s, c in ((0, 1), (3, 100), (7, 255)):
        off = w.C * c * (c - 1) // 2
        M = c * w.C
        want = np.lexsort((np.arange(M), kc[s, :M]))
        got = run.plan.prefix_idx[s * T + off:s * T + off + M].cpu().numpy()
        assert np.array_equal(got, want)
    rng = np.random.default_rng(3)
    rows = np.sort(np.concatenate([rng.choice(w.N, 20, replace=False),
                                   [0, w.C - 1, w.C, w.N - w.C, w.N - 1]]))
    idx = run.idx()
    out = run.out()
    rs = run.rowsum()
    for s in (0, 6):
        q, k, v, gamma, _ = slice_inputs(w, g, s)
        qc = oracle.encode(q, w.bits)
        ref_idx = oracle.select(qc[None], kc[s][None], w.C, w.k, rows=rows)[0]
        assert np.array_equal(idx[s][rows], ref_idx)
        o_ref, s_ref = oracle.attend_fwd(q, k, v, gamma, ref_idx, w.C, rows=rows)
        assert_close_bf16(out[s][rows], o_ref, what="out")
        assert_close_f32(rs[s][rows], s_ref, what="rowsum")


def test_locality_sweep_recall():
    """Selected indices bit-exact for d_K = 1, 2, 3, 8 (21, 42, 30 and 64-bit
    codes); recall against the exact Euclidean top-k falls as d_K grows."""
    rng = np.random.default_rng(4)
    recalls = []
    for w in W.SWEEP:
        w = w.replace(H=2)
        p = zb.problem_of(w)
        g = W.generate(w)
        S = w.B * w.H
        cdt = zb.code_dtype(p)
        qd = torch.from_numpy(g["q"]).cuda().reshape(-1)
        kd = torch.from_numpy(g["k"]).cuda().reshape(-1)
        qc = torch.empty(S * w.N, dtype=cdt, device="cuda")
        kc = torch.empty(S * w.N, dtype=cdt, device="cuda")
        zb.zeta_encode(p, qd, qc)
        zb.zeta_encode(p, kd, kc)
        T = zb.zeta_prefix_entries(p)
        pc = torch.empty(S * T, dtype=cdt, device="cuda")
        pi = torch.empty(S * T, dtype=torch.int32, device="cuda")
        ws = torch.empty(zb.zeta_sort_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        zb.zeta_sort_chunks(p, kc, pc, pi, ws)
        idx = torch.empty(S * w.N * w.k, dtype=torch.int32, device="cuda")
        zb.zeta_select_topk(p, qc, pc, pi, idx)
        torch.cuda.synchronize()
        idx = idx.cpu().numpy().reshape(S, w.N, w.k)
        rows = np.sort(rng.choice(np.arange(w.C, w.N), 96, replace=False))
        hits = []
        for s in range(S):
            b, h = divmod(s, w.H)
            q, k = g["q"][b, h], g["k"][b, h]
            qco, kco = oracle.encode(q, w.bits), oracle.encode(k, w.bits)
            assert np.array_equal(codes_np(qc).reshape(S, w.N)[s], qco)
            ref = oracle.select(qco[None], kco[None], w.C, w.k, rows=rows)[0]
            assert np.array_equal(idx[s][rows], ref)
            exact = oracle.exact_topk(q, k, w.C, w.k, rows=rows)
            hits += [len(set(a.tolist()) & set(e.tolist())) / w.k for a, e in zip(ref, exact)]
        recalls.append(float(np.mean(hits)))
        print(f"recall d_K={w.d_K} bits={w.bits}: {recalls[-1]:.3f}")
    assert all(a > b for a, b in zip(recalls, recalls[1:])), recalls
    assert recalls[0] > 0.8 and recalls[-1] > 0.1
