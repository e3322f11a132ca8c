"""zeta_sort_chunks_noalloc: the sort entry point for callers that cannot
allocate a workspace (it uses the library's fixed device scratch instead).

Its results must equal those of zeta_sort_chunks given a caller-allocated
workspace, call after call, although every call reuses the same scratch."""
import ctypes

import numpy as np
import pytest
import torch

from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem needing more than the 32 MiB scratch is refused on the host
    (ZETA_ERR_WORKSPACE) before anything reaches the GPU."""
    L = zb.lib()
    fn = L.zeta_sort_chunks_noalloc
    fn.argtypes = [ctypes.POINTER(zb.zeta_problem_t)] + [ctypes.c_void_p] * 4
    fn.restype = ctypes.c_int
    big = zb.problem_of(W.TRAIN)                      # ~ 50 MB of sort scratch
    assert zb.zeta_sort_workspace_bytes(big) > 32 << 20
    fake = ctypes.c_void_p(0x1000)
    assert fn(ctypes.byref(big), fake, fake, fake, None) == 3
    bad = zb.problem(1, 1, 1000, 3, 8, 4, 128, 10, "f32")   # C does not divide N
    assert fn(ctypes.byref(bad), fake, fake, fake, None) == 1


def test_noalloc_checks_come_in_the_order_of_the_workspace_sort():
    """zeta_sort_chunks' own checks run before the scratch-size check: more
    than 1024 chunks is ZETA_ERR_UNSUPPORTED even when the problem would also
    need more than 32 MiB, and a problem with nothing to sort (one chunk) is
    ZETA_OK whatever its size, touching nothing."""
    L = zb.lib()
    fn = L.zeta_sort_chunks_noalloc
    fn.argtypes = [ctypes.POINTER(zb.zeta_problem_t)] + [ctypes.c_void_p] * 4
    fn.restype = ctypes.c_int
    fake = ctypes.c_void_p(0x1000)
    many = zb.problem(1, 8, 1 << 22, 3, 64, 16, 2048, 10, "bf16")   # 2048 chunks
    assert zb.zeta_sort_workspace_bytes(many) > 32 << 20
    assert fn(ctypes.byref(many), fake, fake, fake, None) == 2
    one = zb.problem(4, 8, 1 << 20, 3, 64, 16, 1 << 20, 10, "bf16")  # a single chunk
    assert zb.zeta_sort_workspace_bytes(one) > 32 << 20
    assert fn(ctypes.byref(one), fake, fake, fake, None) == 0
    assert L.zeta_sort_chunks(ctypes.byref(one), fake, fake, fake, None, 0, None) == 0


def _sorted_both_ways(w):
    g = W.generate(w)
    p = zb.problem_of(w)
    S, T = w.B * w.H, zb.zeta_prefix_entries(p)
    cdt = zb.code_dtype(p)
    kc = torch.empty(S * w.N, dtype=cdt, device="cuda")
    zb.zeta_encode(p, torch.from_numpy(g["k"]).cuda().reshape(-1), kc)
    ref_c = torch.empty(S * T, dtype=cdt, device="cuda")
    ref_i = torch.empty(S * T, dtype=torch.int32, device="cuda")
    ws = torch.empty(zb.zeta_sort_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    zb.zeta_sort_chunks(p, kc, ref_c, ref_i, ws)
    got_c = torch.full((S * T,), -1, dtype=cdt, device="cuda")
    got_i = torch.full((S * T,), -1, dtype=torch.int32, device="cuda")
    zb.zeta_sort_chunks_noalloc(p, kc, got_c, got_i)
    torch.cuda.synchronize()
    return ref_c.cpu().numpy(), ref_i.cpu().numpy(), got_c.cpu().numpy(), got_i.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_sort_matches_workspace_sort_on_consecutive_calls():
    """Two calls in a row (different sizes and inputs, the second smaller, so
    stale scratch from the first is present) give exactly the workspace
    version's prefix tables."""
    first = W.EFFICIENCY.replace(H=4)                      # ~ 10 MB of scratch
    second = W.CLUSTERED.replace(seed=5)
    for w in (first, second):
        p = zb.problem_of(w)
        assert zb.zeta_sort_workspace_bytes(p) <= 32 << 20
        rc, ri, gc, gi = _sorted_both_ways(w)
        assert np.array_equal(gi, ri)
        assert np.array_equal(gc, rc)
