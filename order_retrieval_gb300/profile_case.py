"""Run whole ZETA steps on one workload, for profilers (ncu) and quick timing.

  python -m order_retrieval_gb300.profile_case [--workload NAME] [--B B] \
      [--steps K] [--warmup W] [--fwd-only]

Each step enqueues encode (q, k), sort, select, attend forward and (unless
--fwd-only) attend backward through the C ABI, then synchronises.  Prints the
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
    a = ap.parse_args()
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


if __name__ == "__main__":
    main()
