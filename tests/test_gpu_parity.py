"""GPU parity: the CUDA library (called through its C ABI) against the CPU oracle.

Integer results (codes, prefix tables, selected indices) must match bit for
bit.  Floating-point results use the stated tolerances: float32 tensors
max |x - x_ref| <= 1e-5 (relative above magnitude 1); bf16 tensors
max |x - x_ref| <= 2e-2 * max |x_ref| with the oracle fed the same
bf16-rounded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W

from gpu_util import (Run, assert_close_bf16, assert_close_f32, codes_np, dev_vals,
                      host_vals, in_threads, slice_inputs)

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def _prefix_is_sorted_permutation(pc, pi, w):
    """Property check of a whole prefix table: each prefix c is a permutation
    of 0..cC-1 sorted by (code, index)."""
    for c in range(1, w.n_chunks):
        off = w.C * c * (c - 1) // 2
        M = c * w.C
        codes = pc[off:off + M]
        idx = pi[off:off + M].astype(np.int64)
        assert np.array_equal(np.sort(idx), np.arange(M))
        key = codes.astype(np.uint64)
        assert (key[1:] >= key[:-1]).all()
        tie = key[1:] == key[:-1]
        assert (idx[1:][tie] > idx[:-1][tie]).all()


def _check_forward_host(w, g, s, idx_s, out_s, rs_s, rows=None, bf16=False):
    """Slice s of a forward (device results already on the host, all N rows)
    against the oracle: idx bit for bit, rowsum at float32, out at the
    tolerance of its dtype; rows limits the check to those queries."""
    q, k, v, gamma, _ = slice_inputs(w, g, s)
    qc = oracle.encode(q, w.bits)
    kc = oracle.encode(k, w.bits)
    idx_ref = oracle.select(qc[None], kc[None], w.C, w.k, rows=rows)[0]
    sel = slice(None) if rows is None else rows
    assert np.array_equal(idx_s[sel], idx_ref)
    out_ref, rs_ref = oracle.attend_fwd(q, k, v, gamma, idx_ref, w.C, rows=rows)
    assert_close_f32(rs_s[sel], rs_ref, what="rowsum")
    if bf16:
        assert_close_bf16(out_s[sel], out_ref, what="out")
    else:
        assert_close_f32(out_s[sel], out_ref, what="out")


def _check_forward_slice(run, s, rows=None, bf16=False):
    _check_forward_host(run.w, run.g, s, run.idx()[s], run.out()[s], run.rowsum()[s], rows, bf16)


# ------------------------------------------------------------------ encode ---

@pytest.mark.parametrize("w", [W.TINY, W.CLUSTERED, *W.SWEEP], ids=lambda w: w.name)
def test_encode_bit_exact(w):
    run_w = w.replace(B=1, H=2) if w.B * w.H > 2 else w
    g = W.generate(run_w)
    p = zb.problem_of(run_w)
    for name in ("q", "k"):
        x = torch.from_numpy(g[name]).cuda().reshape(-1)
        codes = torch.empty(run_w.B * run_w.H * run_w.N, dtype=zb.code_dtype(p), device="cuda")
        zb.zeta_encode(p, x, codes)
        torch.cuda.synchronize()
        assert np.array_equal(codes_np(codes), oracle.encode(g[name], run_w.bits).reshape(-1))


@pytest.mark.parametrize("d_K,bits", [(1, 24), (2, 21), (3, 10), (3, 12), (8, 8), (5, 12)])
def test_encode_edge_values(d_K, bits):
    """Grid edges, clamping, NaN and infinities."""
    half = 2.0 ** (bits - 1)
    vals = [-1.0, -1.0 + 1 / half, -0.5, 0.0, 1 / half, 0.999, np.nextafter(np.float32(1), 0),
            1.0, 5.0, -7.0, np.nan, np.inf, -np.inf, -1.0 - 1e-7, 2.0 ** -30]
    vals = np.array(vals, dtype=np.float32)
    rng = np.random.default_rng(d_K * 100 + bits)
    x = rng.choice(vals, size=(1, 1, 4096, d_K)).astype(np.float32)
    p = zb.problem(1, 1, 4096, d_K, 8, 1, 4096, bits, "f32")
    codes = torch.empty(4096, dtype=zb.code_dtype(p), device="cuda")
    zb.zeta_encode(p, torch.from_numpy(x).cuda().reshape(-1), codes)
    torch.cuda.synchronize()
    assert np.array_equal(codes_np(codes), oracle.encode(x, bits).reshape(-1))


# ---------------------------------------------------------- sort / select ---

@pytest.mark.parametrize("w", [W.TINY, W.CLUSTERED], ids=lambda w: w.name)
def test_prefix_and_select_bit_exact(w):
    run = Run(w)
    g = run.g
    qc = oracle.encode(g["q"], w.bits).reshape(run.S, w.N)
    kc = oracle.encode(g["k"], w.bits).reshape(run.S, w.N)
    assert np.array_equal(run.q_codes(), qc)
    assert np.array_equal(run.k_codes(), kc)
    pc_ref, pi_ref = oracle.prefix_table(kc, w.C)
    pc, pi = run.prefix()
    assert np.array_equal(pi, pi_ref)
    assert np.array_equal(pc, pc_ref)
    assert np.array_equal(run.idx(), oracle.select(qc, kc, w.C, w.k))


# ----------------------------------------------------------------- forward ---

def test_forward_tiny_f32():
    run = Run(W.TINY)
    assert run.status() == 0
    _check_forward_slice(run, 0)


def test_forward_clustered_bf16():
    run = Run(W.CLUSTERED)
    assert run.status() == 0
    for s in range(run.S):
        _check_forward_slice(run, s, bf16=True)


@pytest.mark.parametrize("w", [W.EFFICIENCY, W.PAGES12], ids=lambda w: w.name)
def test_forward_efficiency_sampled(w):
    """The 65,536-token workload in the timed launch configuration (and with
    the pages' 12-bit grid, 36-bit codes in 64-bit containers): prefix tables
    of every slice checked by property, one slice's table exactly, and sampled
    queries of every slice against the oracle."""
    run = Run(w)
    assert run.status() == 0
    g = run.g
    kc_ref = oracle.encode(g["k"], w.bits).reshape(run.S, w.N)
    qc_ref = oracle.encode(g["q"], w.bits).reshape(run.S, w.N)
    assert np.array_equal(run.k_codes(), kc_ref)
    assert np.array_equal(run.q_codes(), qc_ref)
    pc, pi = run.prefix()
    for s in range(run.S):
        _prefix_is_sorted_permutation(pc[s], pi[s], w)
    for c in (1, 2, 31, 63):
        off = w.C * c * (c - 1) // 2
        M = c * w.C
        want = np.lexsort((np.arange(M), kc_ref[3, :M]))
        assert np.array_equal(pi[3, off:off + M], want)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([rng.choice(w.N, 120, replace=False),
                                   [0, w.C - 1, w.C, 2 * w.C - 1, w.N - 1]]))
    idx, out, rs = run.idx(), run.out(), run.rowsum()
    # slice 5 whole, element by element; the other slices on the sampled rows
    cases = [(s, None if s == 5 else rows) for s in range(run.S)]
    in_threads(lambda c: _check_forward_host(w, g, c[0], idx[c[0]], out[c[0]], rs[c[0]],
                                             rows=c[1], bf16=True), cases)


# ---------------------------------------------------------------- backward ---

def _oracle_idx(run, s):
    """The oracle's own selection for slice s (the backward's fixed input),
    checked against the device selection once and cached on the run."""
    cache = run.__dict__.setdefault("_idx_ref", {})
    if s not in cache:
        w = run.w
        q, k, _, _, _ = slice_inputs(w, run.g, s)
        ref = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None],
                            w.C, w.k)[0]
        assert np.array_equal(run.idx()[s], ref)
        cache[s] = ref
    return cache[s]


def _check_backward_slice(run, s, bf16=False):
    w, g = run.w, run.g
    q, k, v, gamma, dout = slice_inputs(w, g, s)
    idx = _oracle_idx(run, s)
    dq_r, dk_r, dv_r, _ = oracle.attend_bwd(q, k, v, gamma, idx, dout, w.C)
    dq, dk, dv, _ = run.grads()
    if bf16:
        assert_close_bf16(dq[s], dq_r, what="dq")
        assert_close_bf16(dk[s], dk_r, what="dk")
        assert_close_bf16(dv[s], dv_r, what="dv")
    else:
        assert_close_f32(dq[s], dq_r, what="dq")
        assert_close_f32(dk[s], dk_r, what="dk")
        assert_close_f32(dv[s], dv_r, what="dv")


def _dgamma_ref(run):
    w, g = run.w, run.g
    ref = np.zeros(w.H)
    for s in range(run.S):
        q, k, v, gamma, dout = slice_inputs(w, g, s)
        ref[s % w.H] += oracle.attend_bwd(q, k, v, gamma, _oracle_idx(run, s), dout, w.C)[3]
    return ref


def test_backward_tiny_f32():
    run = Run(W.TINY, backward=True)
    assert run.status() == 0
    _check_backward_slice(run, 0)
    dg = run.grads()[3]
    assert_close_f32(dg, _dgamma_ref(run), what="dgamma")


def test_backward_fd_workload_f32():
    w = W.FD.replace(v_dtype="f32")
    run = Run(w, backward=True)
    for s in range(run.S):
        _check_backward_slice(run, s)
    assert_close_f32(run.grads()[3], _dgamma_ref(run), what="dgamma")


def _train_slices_against_oracle(run, full, head, bf16):
    """The training workload's backward: dq, dk, dv of the slices in `full`
    element by element, and dgamma of `head`, which sums over that head's B
    slices s = b*H + head, against the sum of the oracle's per-slice values.
    Each slice's selection comes from the oracle (checked against the device's
    bit for bit); the oracle runs on all listed slices at once in threads."""
    w, g = run.w, run.g
    hs = [b * w.H + head for b in range(w.B)]
    todo = sorted(set(full) | set(hs))
    dev_idx = {s: run.idx_slice(s) for s in todo}

    def one(s):
        q, k, v, gamma, dout = slice_inputs(w, g, s)
        ref = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None],
                            w.C, w.k)[0]
        assert np.array_equal(dev_idx[s], ref), f"idx of slice {s}"
        return oracle.attend_bwd(q, k, v, gamma, ref, dout, w.C)

    refs = dict(zip(todo, in_threads(one, todo)))
    close = assert_close_bf16 if bf16 else assert_close_f32
    for s in full:
        dq, dk, dv = run.grads_slice(s)
        dq_r, dk_r, dv_r, _ = refs[s]
        close(dq, dq_r, what=f"dq[{s}]")
        close(dk, dk_r, what=f"dk[{s}]")
        close(dv, dv_r, what=f"dv[{s}]")
    dg = run.plan.dgamma.cpu().numpy().astype(np.float64)
    dg_ref = sum(refs[s][3] for s in hs)
    close(np.array([dg[head]]), np.array([dg_ref]), what=f"dgamma[{head}]")


def test_backward_train_f32_sampled():
    """The training workload (B=4, H=8, N=65536, k=48, C=1024) with float32
    values and upstream gradients: slices 0 and 29 whole, and the gamma
    gradient of head 5 (slices 5, 13, 21, 29) against the oracle."""
    w = W.TRAIN.replace(v_dtype="f32")
    run = Run(w, backward=True)
    assert run.status() == 0
    _train_slices_against_oracle(run, full=(0, 29), head=5, bf16=False)


def test_backward_train_bf16_sampled():
    """The timed training workload itself (bf16 values and dO, tensor-core
    kernels): slices 0 and 31 whole, and the gamma gradient of head 7
    (slices 7, 15, 23, 31) against the oracle."""
    run = Run(W.TRAIN, backward=True)
    assert run.status() == 0
    _train_slices_against_oracle(run, full=(0, 31), head=7, bf16=True)


def test_backward_beyond_float_slot_division():
    """N k above 2^24 (N = 65536, k = 260): the backward's transpose maps a
    window slot to its query by integer division instead of the float
    reciprocal; one slice against the oracle."""
    w = W.TRAIN.replace(name="train_k260", B=1, H=1, k=260)
    assert w.N * w.k > 1 << 24
    run = Run(w, backward=True)
    assert run.status() == 0
    _check_backward_slice(run, 0, bf16=True)
    assert_close_bf16(run.grads()[3], _dgamma_ref(run), what="dgamma")


def test_backward_train_one_batch_bf16():
    """One batch of the training workload (H=8, N=65536, k=48, C=1024; about
    1 GB on the device): slices 0 and 7 whole and the gamma gradient of every
    head against the oracle."""
    w = W.TRAIN.replace(name="train_bf16_b1_n65536", B=1)
    run = Run(w, backward=True)
    assert run.status() == 0
    refs = {}

    def one(s):
        q, k, v, gamma, dout = slice_inputs(w, run.g, s)
        ref = oracle.select(oracle.encode(q, w.bits)[None], oracle.encode(k, w.bits)[None],
                            w.C, w.k)[0]
        return ref, oracle.attend_bwd(q, k, v, gamma, ref, dout, w.C)

    res = in_threads(one, range(run.S))
    dev_idx = run.idx()
    for s, (ref_idx, r) in enumerate(res):
        assert np.array_equal(dev_idx[s], ref_idx)
        refs[s] = r
    for s in (0, 7):
        dq, dk, dv = run.grads_slice(s)
        assert_close_bf16(dq, refs[s][0], what="dq")
        assert_close_bf16(dk, refs[s][1], what="dk")
        assert_close_bf16(dv, refs[s][2], what="dv")
    dg = run.plan.dgamma.cpu().numpy().astype(np.float64)
    assert_close_bf16(dg, np.array([refs[s][3] for s in range(run.S)]), what="dgamma")


def test_backward_beyond_16bit_sequence_bf16():
    """N = 131072 (> 2^16) takes the unpacked (key, query) transpose in the
    tensor-core backward; one slice against the oracle."""
    w = W.TRAIN.replace(name="train_n131072", B=1, H=1, N=131072, C=512, k=16)
    run = Run(w, backward=True)
    assert run.status() == 0
    _check_backward_slice(run, 0, bf16=True)


def test_backward_clustered_bf16():
    w = W.CLUSTERED.replace(B=1)
    run = Run(w, backward=True)
    assert run.status() == 0
    for s in (0, 5):
        _check_backward_slice(run, s, bf16=True)


def test_backward_is_deterministic():
    w = W.CLUSTERED.replace(B=1, H=2)
    a = Run(w, backward=True)
    ga = [t.copy() for t in a.grads()]
    a.plan.backward(a.q, a.k, a.v, a.gamma, a.dout)
    torch.cuda.synchronize()
    for x, y in zip(ga, a.grads()):
        assert np.array_equal(x, y)


# -------------------------------------------------------------- edge cases ---

EDGE = [
    dict(N=96, C=32, k=32, d_V=8),          # k = C, ragged tiles
    dict(N=200, C=40, k=7, d_V=40),         # odd k, d_V not a multiple of 32
    dict(N=256, C=256, k=16),               # one chunk: everything is local
    dict(N=512, C=64, k=8, bits=1),         # 3-bit codes: massive ties
    dict(N=512, C=16, k=16, d_V=1),         # many chunks, d_V = 1
    dict(N=384, C=128, k=5, d_K=1, bits=21),
    dict(N=384, C=128, k=9, d_K=2, bits=21),   # 42-bit codes
    dict(N=384, C=128, k=12, d_K=8, bits=8),   # 64-bit codes
    dict(N=4096, C=4, k=4, d_V=16),         # 1024 chunks (the limit)
]


@pytest.mark.parametrize("kw", EDGE, ids=lambda kw: "-".join(f"{a}{b}" for a, b in kw.items()))
@pytest.mark.parametrize("vd", ["f32", "bf16"])
def test_edge_shapes(kw, vd):
    base = dict(name="edge", B=1, H=2, N=256, d_K=3, d_V=32, k=8, C=64, bits=10, v_dtype=vd,
                gamma=(0.3, 1.0), dist="uniform", v_dist="normal", seed=11)
    base.update(kw)
    w = W.Workload(**base)
    run = Run(w, backward=True)
    assert run.status() == 0
    g = run.g
    qc = oracle.encode(g["q"], w.bits).reshape(run.S, w.N)
    kc = oracle.encode(g["k"], w.bits).reshape(run.S, w.N)
    if w.n_chunks > 1:
        pc_ref, pi_ref = oracle.prefix_table(kc, w.C)
        pc, pi = run.prefix()
        assert np.array_equal(pi, pi_ref)
        assert np.array_equal(pc, pc_ref)
    assert np.array_equal(run.idx(), oracle.select(qc, kc, w.C, w.k))
    for s in range(run.S):
        _check_forward_slice(run, s, bf16=(vd == "bf16"))
        _check_backward_slice(run, s, bf16=(vd == "bf16"))
    ref = _dgamma_ref(run)
    if vd == "bf16":
        assert_close_bf16(run.grads()[3], ref, what="dgamma")
    else:
        assert_close_f32(run.grads()[3], ref, what="dgamma")


TC = [
    dict(N=200, C=40, k=7),                 # chunks shorter than a query tile
    dict(N=300, C=60, k=12),                # C not a multiple of 8: transpose sorted by key
    dict(N=480, C=96, k=33),                # one full tile plus a ragged one, k > 32
    dict(N=256, C=256, k=16),               # a single chunk: all local, four tiles
    dict(N=1024, C=128, k=128, d_K=1, bits=20),
    dict(N=768, C=192, k=64, d_K=2, bits=12),
    dict(N=512, C=128, k=20, d_K=4, bits=6),
    dict(N=512, C=64, k=64, bits=1),        # heavy code ties
    # the key side's own-chunk kernel (C a multiple of 128): an odd number of
    # one-tile units, d_K = 2, and more heads than its gamma table (H = 65: the
    # key kernel then computes the own-chunk block itself)
    dict(B=1, H=1, N=384, C=128, k=16),
    dict(N=512, C=128, k=20, d_K=2, bits=12),
    dict(B=1, H=65, N=256, C=128, k=8),
    dict(N=768, C=384, k=16),               # three key tiles per chunk (pairs span chunks)
    dict(B=1, H=2, N=8192, C=4096, k=64),   # units of up to 32 query tiles
]


@pytest.mark.parametrize("kw", TC, ids=lambda kw: "-".join(f"{a}{b}" for a, b in kw.items()))
def test_tensor_core_path(kw):
    """bf16 values with d_V = 64 run the tensor-core forward and backward;
    ragged tiles, k up to C, d_K from 1 to 4, the key side's own-chunk block
    on tcgen05 and its fallback, and the backward's transpose sorted by 8-key
    group (C a multiple of 8) or by key."""
    base = dict(name="tc", B=2, H=2, N=256, d_K=3, d_V=64, k=8, C=64, bits=10, v_dtype="bf16",
                gamma=(0.3, 1.0), dist="uniform", v_dist="normal", seed=21)
    base.update(kw)
    w = W.Workload(**base)
    run = Run(w, backward=True)
    assert run.status() == 0
    for s in range(run.S):
        _check_forward_slice(run, s, bf16=True)
        _check_backward_slice(run, s, bf16=True)
    assert_close_bf16(run.grads()[3], _dgamma_ref(run), what="dgamma")


def test_values_not_32_byte_aligned():
    """v at a 16-byte but not 32-byte boundary: the tensor-core forward reads
    value rows 32 bytes at a time, so the two-call and the fused forward both
    take the general kernel; their results match the oracle."""
    w = W.Workload(name="tc", B=1, H=2, N=512, d_K=3, d_V=64, k=16, C=128, bits=10,
                   v_dtype="bf16", gamma=(0.3, 1.0), dist="uniform", v_dist="normal", seed=23)
    run = Run(w)
    pl = run.plan
    buf = torch.empty(run.v.numel() + 8, dtype=torch.bfloat16, device="cuda")
    v16 = buf[8:]
    v16.copy_(run.v)
    assert v16.data_ptr() % 32 == 16
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, rowsum = torch.empty_like(pl.out), torch.empty_like(pl.rowsum)
    zb.zeta_attend_fwd(run.p, run.q, run.k, v16, run.gamma, pl.idx, out, rowsum, status)
    idx2 = torch.empty_like(pl.idx)
    out2, rowsum2 = torch.empty_like(pl.out), torch.empty_like(pl.rowsum)
    zb.zeta_select_attend_fwd(run.p, run.q, run.k, v16, run.gamma, pl.q_codes, pl.prefix_codes,
                              pl.prefix_idx, idx2, out2, rowsum2, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for o, rs, ix in ((out, rowsum, pl.idx), (out2, rowsum2, idx2)):
        o_h = host_vals(o).reshape(run.S, run.N, w.d_V)
        rs_h = rs.cpu().numpy().astype(np.float64).reshape(run.S, run.N)
        ix_h = ix.cpu().numpy().reshape(run.S, run.N, w.k)
        for s in range(run.S):
            _check_forward_host(w, run.g, s, ix_h[s], o_h[s], rs_h[s], bf16=True)


def test_empty_problem_is_a_no_op():
    p = zb.problem(1, 2, 0, 3, 32, 8, 64, 10, "f32")
    x = torch.empty(0, device="cuda")
    codes = torch.empty(0, dtype=torch.int32, device="cuda")
    zb.zeta_encode(p, x, codes)
    torch.cuda.synchronize()


def test_out_of_range_indices_are_flagged_and_skipped():
    w = W.TINY.replace(N=256, C=64, k=8)
    g = W.generate(w)
    run = Run(w)
    idx = run.plan.idx.clone()
    bad = idx.view(w.N, w.k)
    bad[100, 0] = 200            # a key of the query's own chunk or later: illegal
    bad[150, 3] = -5
    bad[255, 7] = 10_000_000
    out = torch.empty_like(run.plan.out)
    rs = torch.empty_like(run.plan.rowsum)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zb.zeta_attend_fwd(run.p, run.q, run.k, run.v, run.gamma, idx, out, rs, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 6
    ref_idx = bad.cpu().numpy().copy()
    ref_idx[100, 0] = ref_idx[150, 3] = ref_idx[255, 7] = -1
    q, k, v, gamma, _ = slice_inputs(w, g, 0)
    o_ref, s_ref = oracle.attend_fwd(q, k, v, gamma, ref_idx, w.C)
    assert_close_f32(out.cpu().numpy().reshape(w.N, w.d_V), o_ref, what="out")
    assert_close_f32(rs.cpu().numpy(), s_ref, what="rowsum")
