"""Run whole ZETA steps on one workload, for profilers (ncu) and quick timing.

  python -m order_retrieval_gb300.profile_case [--workload NAME] [--B B] \
      [--steps K] [--warmup W] [--fwd-only] [--projection]

Each step enqueues encode (q, k), sort, select, attend forward and (unless
--fwd-only) attend backward through the C ABI, then synchronises.  With
--projection a step is the fused two-layer projection + encode alone on the
projection workload (B=4, N=65536, D=512 unless --B is given).  Prints the
mean step time measured with CUDA events.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import binding as zb
from . import workloads as W
from .pipeline import ZetaPlan


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=W.TRAIN.name, choices=sorted(W.ALL))
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--projection", action="store_true")
    a = ap.parse_args()
    if a.projection:
        return projection(a)
    w = W.ALL[a.workload]
    if a.B is not None:
        w = w.replace(B=a.B)
    g = W.generate(w, with_dout=not a.fwd_only)
    p = zb.problem_of(w)

    def dev(x, vals=False):
        t = torch.from_numpy(np.ascontiguousarray(x)).reshape(-1)
        if vals and x.dtype == np.int16:
            t = t.view(torch.bfloat16)
        return t.cuda()

    q, k, v, gamma = dev(g["q"]), dev(g["k"]), dev(g["v"], True), dev(g["gamma"])
    dout = None if a.fwd_only else dev(g["dout"], True)
    plan = ZetaPlan(p, "cuda", backward=not a.fwd_only)

    def step():
        plan.forward(q, k, v, gamma)
        if dout is not None:
            plan.backward(q, k, v, gamma, dout)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    ts = []
    for _ in range(a.steps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        step()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    if int(plan.status.item()) != 0:
        raise SystemExit(f"device status {plan.status.item()}")
    print(f"{w.name} B={w.B} step_ms={sum(ts) / len(ts):.3f}")


def projection(a):
    pj = W.PROJ
    if a.B is not None:
        pj = W.Projection(pj.name, pj.base.replace(B=a.B), pj.D, pj.F, pj.seed)
    w = pj.base
    g = W.generate_projection(pj)
    p = zb.problem_of(w)

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x)).view(torch.bfloat16).reshape(-1).cuda()

    x, w1 = bf(g["x"]), bf(g["W1"])
    b1, w2, b2 = (torch.from_numpy(g[n]).reshape(-1).cuda() for n in ("b1", "W2", "b2"))
    S = w.B * w.H * w.N
    q = torch.empty(S * w.d_K, dtype=torch.float32, device="cuda")
    k = torch.empty_like(q)
    qc = torch.empty(S, dtype=zb.code_dtype(p), device="cuda")
    kc = torch.empty_like(qc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        zb.zeta_project_encode(p, pj.D, pj.F, x, w1, b1, w2, b2, q, k, qc, kc, st)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    ts = []
    for _ in range(a.steps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        step()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    if int(st.item()) != 0:
        raise SystemExit(f"device status {st.item()}")
    flop = 2.0 * w.B * w.N * pj.D * 2 * w.H * pj.F
    ms = sum(ts) / len(ts)
    print(f"{pj.name} B={w.B} kernel_ms={ms:.4f} tflops={flop / ms / 1e9:.1f}")


if __name__ == "__main__":
    main()
