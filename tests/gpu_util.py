"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, bring results back as numpy."""
import concurrent.futures as cf
import os

import numpy as np
import torch

from order_retrieval_gb300 import binding as zb
from order_retrieval_gb300 import workloads as W


def dev_vals(w, arr):
    """float32 array or bf16 bit patterns -> CUDA tensor of the workload dtype."""
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if arr.dtype == np.int16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def host_vals(t):
    """CUDA float32 / bf16 tensor -> float64 numpy."""
    if t.dtype == torch.bfloat16:
        return W.bf16_bits_to_f32(t.view(torch.int16).cpu().numpy()).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def codes_np(t):
    a = t.cpu().numpy()
    return a.view(np.uint32).astype(np.uint64) if a.dtype == np.int32 else a.view(np.uint64)


class Run:
    """Device tensors and results of one forward (and optional backward)."""

    def __init__(self, w, g=None, backward=False, dout=None, weight="cauchy"):
        self.w = w
        self.g = g if g is not None else W.generate(w, with_dout=backward)
        self.p = zb.problem_of(w, weight=weight)
        S, N = w.B * w.H, w.N
        self.q = torch.from_numpy(self.g["q"]).cuda().reshape(-1)
        self.k = torch.from_numpy(self.g["k"]).cuda().reshape(-1)
        self.v = dev_vals(w, self.g["v"]).reshape(-1)
        self.gamma = torch.from_numpy(self.g["gamma"]).cuda()
        from order_retrieval_gb300.pipeline import ZetaPlan
        self.plan = ZetaPlan(self.p, "cuda", backward=backward)
        self.plan.forward(self.q, self.k, self.v, self.gamma)
        if backward:
            d = self.g["dout"] if dout is None else dout
            self.dout = dev_vals(w, d).reshape(-1)
            self.plan.backward(self.q, self.k, self.v, self.gamma, self.dout)
        torch.cuda.synchronize()
        self.S, self.N = S, N

    # results as numpy, [S, ...]
    def q_codes(self):
        return codes_np(self.plan.q_codes).reshape(self.S, self.N)

    def k_codes(self):
        return codes_np(self.plan.k_codes).reshape(self.S, self.N)

    def prefix(self):
        T = self.plan.T
        return (codes_np(self.plan.prefix_codes).reshape(self.S, T),
                self.plan.prefix_idx.cpu().numpy().reshape(self.S, T))

    def idx(self):
        return self.plan.idx.cpu().numpy().reshape(self.S, self.N, self.w.k)

    def out(self):
        return host_vals(self.plan.out).reshape(self.S, self.N, self.w.d_V)

    def rowsum(self):
        return self.plan.rowsum.cpu().numpy().astype(np.float64).reshape(self.S, self.N)

    def status(self):
        return int(self.plan.status.item())

    def idx_slice(self, s):
        return self.plan.idx.view(self.S, self.N, self.w.k)[s].cpu().numpy()

    def grads_slice(self, s):
        """(dq, dk, dv) of slice s as float64 numpy."""
        w = self.w
        return (self.plan.dq.view(self.S, self.N, w.d_K)[s].cpu().numpy().astype(np.float64),
                self.plan.dk.view(self.S, self.N, w.d_K)[s].cpu().numpy().astype(np.float64),
                host_vals(self.plan.dv.view(self.S, self.N, w.d_V)[s]))

    def grads(self):
        w = self.w
        return (self.plan.dq.cpu().numpy().astype(np.float64).reshape(self.S, self.N, w.d_K),
                self.plan.dk.cpu().numpy().astype(np.float64).reshape(self.S, self.N, w.d_K),
                host_vals(self.plan.dv).reshape(self.S, self.N, w.d_V),
                self.plan.dgamma.cpu().numpy().astype(np.float64))


def slice_inputs(w, g, s):
    """Oracle inputs of slice s (float64 values, bf16 already widened)."""
    b, h = divmod(s, w.H)
    q = g["q"][b, h]
    k = g["k"][b, h]
    v = W.values_f64(w, g["v"][b, h])
    gamma = float(g["gamma"][h])
    dout = W.values_f64(w, g["dout"][b, h]) if "dout" in g else None
    return q, k, v, gamma, dout


def assert_close_bf16(got, ref, rel=2e-2, what=""):
    """bf16 criterion: max |got - ref| <= rel * max |ref| over the tensor."""
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    assert err <= rel * scale, f"{what}: max err {err:.3e} > {rel} * {scale:.3e}"


def assert_close_f32(got, ref, atol=1e-5, what=""):
    """fp32 criterion: max |got - ref| <= 1e-5, relative above magnitude 1."""
    err = np.abs(got - ref)
    bound = atol * np.maximum(1.0, np.abs(ref))
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} entries off, worst {err.max():.3e}"


def in_threads(fn, items):
    """fn over items on every host core; the oracle's C calls release the GIL,
    so threads run them in parallel.  Results in the order of items."""
    items = list(items)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(items), os.cpu_count() or 1))) as ex:
        return list(ex.map(fn, items))
