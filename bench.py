"""Benchmark of the ZETA hot path (prints one JSON line on rank 0).

One step = the whole path over one batch: Z-order encode of q and k, sorted
causal prefixes, window select, Cauchy attend forward and backward, on the
training workload (B=4, H=8, N=65536, d_K=3, d_V=64, k=48, C=1024, 10 bits,
bf16 values).  `value` is forward+backward tokens/s (B*N per step) with inputs
resident in HBM; the forward alone is also timed on that workload and on the
efficiency workload (B=1, H=8, N=65536, k=64), whose attend-forward kernel
carries the HBM roofline figure.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The 1,048,576-token workload (B=1, H=8, k=64, C=4096) is timed forward only,
and the peak device memory of each workload is reported.

--impl reference times the CPU oracle (single thread) on a bounded sample of
the same workload: the queries of two chunks of one full-length slice.  Under
torchrun every rank runs its own batch (weak scaling) and the gamma gradient is
summed across ranks (the only exchange the path has).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# forward attend kernel on the efficiency workload, from one ncu capture, with a
# digest of the kernel's sources at that time.  The line reports the figure only
# while the sources still have that digest (else null: the kernel has changed).
ATTEND_FWD_TRAFFIC = {
    "bytes": 211_883_264 + 50_172_928,
    "sources_sha256": "1f869ed914bf2ba294714b0d28c1e84d3f46bcaaf494aefeeb24e33843656388",
    "capture": "attend_fwd_tc, efficiency_bf16_n65536, ncu --metrics "
               "dram__bytes_read.sum,dram__bytes_write.sum",
}
ATTEND_FWD_SOURCES = ("attend_fwd_tc.cu", "attend_fwd_tc.cuh", "mma.cuh", "common.cuh")

METRIC = "ZETA attention tokens/s (fwd, fwd+bwd) at N=65536 and % of GB300 HBM roofline"
L2_FLUSH_BYTES = 256 << 20
PAGES_FWD_MB = 17348.2        # the pages' forward memory at 65,536 tokens (context)


def sources_digest(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "order_retrieval_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------ byte models ---

def fwd_attend_bytes(w) -> int:
    """Algorithmic bytes of one attend-forward launch: per query, the k window
    rows of v (d_V values) and k (d_K floats) and their indices, its own q, its
    output row and row sum; per key, its own-chunk k and v row once."""
    vb = 2 if w.v_dtype == "bf16" else 4
    rows = w.B * w.H * w.N
    per_q = w.k * (w.d_V * vb + w.d_K * 4 + 4) + w.d_K * 4 + w.d_V * vb + 4
    per_key_local = w.d_K * 4 + w.d_V * vb
    return rows * (per_q + per_key_local)


def fused_fwd_bytes(w) -> int:
    """Algorithmic bytes of one fused select + attend launch: the attend
    forward's bytes (the window read from the sorted prefix in place of an
    index row), plus per query its code, the binary-search probes (one code per
    halving of its prefix) and the index row written for the backward."""
    rows = w.B * w.H * w.N
    cb = 4 if w.d_K * w.bits <= 32 else 8
    probes = max(1, (w.N - w.C).bit_length())
    return fwd_attend_bytes(w) + rows * (cb + probes * cb + 4 * w.k)


def bwd_attend_bytes(w) -> int:
    """Algorithmic bytes of one attend-backward call: per query, the window v
    rows again (query side) and the window dO rows gathered on the key side,
    window k / q rows, indices read twice plus the transpose (read + write),
    dO, dq; per key, own-chunk k, v, dO rows, dk, dv."""
    vb = 2 if w.v_dtype == "bf16" else 4
    rows = w.B * w.H * w.N
    per_q = (w.k * (2 * w.d_V * vb + 2 * w.d_K * 4 + 4 * 4)
             + w.d_V * vb + 2 * w.d_K * 4 + 16)
    per_key = 3 * (w.d_K * 4 + w.d_V * vb) + w.d_K * 4 + w.d_V * vb
    return rows * (per_q + per_key)


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t is not None:
                self.t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def physical_gpu_index(local: int) -> int:
    """nvidia-smi index of this process's GPU (CUDA_VISIBLE_DEVICES aware)."""
    vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    if local < len(vis) and vis[local].isdigit():
        return int(vis[local])
    return local


# ------------------------------------------------------------ reference arm ---

def cpu_slice(w):
    """Oracle inputs of one (b, h) slice of the workload at its full length N:
    the generator's draw of a one-slice version of the workload (same
    distribution and sizes, its own random values)."""
    from order_retrieval_gb300 import workloads as W
    g = W.generate(w.replace(B=1, H=1), with_dout=True)
    q, k = g["q"][0, 0], g["k"][0, 0]
    v = W.values_f64(w, g["v"][0, 0])
    do = W.values_f64(w, g["dout"][0, 0])
    return q, k, v, do, float(g["gamma"][0])


def sample_rows(w):
    """The queries of two chunks placed symmetrically about the middle of the
    sequence (chunks n/4 and 3n/4 - 1 of n).  The oracle's work per query is
    constant in the attend steps and linear in the chunk index in its select
    (a count over the prefix), so the mean cost per query of the pair is the
    mean over the whole slice."""
    n = w.N // w.C
    cs = sorted({n // 4, max(0, 3 * n // 4 - 1)})
    return np.concatenate([np.arange(c * w.C, (c + 1) * w.C) for c in cs])


def oracle_step(w, sample, rows=None):
    """The oracle's path on one slice: encode, select, attend forward and
    backward, for every query (rows None) or the listed ones."""
    import oracle
    q, k, v, do, gamma = sample
    qc = oracle.encode(q, w.bits)
    kc = oracle.encode(k, w.bits)
    idx = oracle.select(qc[None], kc[None], w.C, w.k, rows=rows)[0]
    oracle.attend_fwd(q, k, v, gamma, idx, w.C, rows=rows)
    oracle.attend_bwd(q, k, v, gamma, idx, do, w.C, rows=rows)


def oracle_tokens_per_s(w, queries: int, seconds: float) -> float:
    """A slice's queries belong to one of H heads: H of them make one token of
    the metric (B*N tokens per step)."""
    return queries / w.H / seconds


def _oracle_shard(wname):
    """One host core's share of the sharded CPU baseline (a spawned process;
    no GPU work): draws its slice, then times the oracle on it."""
    from order_retrieval_gb300 import workloads as W
    w = W.ALL[wname]
    sample = cpu_slice(w)
    t0 = time.perf_counter()
    oracle_step(w, sample)
    return time.perf_counter() - t0


def cpu_sharded(w):
    """The oracle on every host core at once, one spawned process per core,
    each on a full slice; slices are independent, so this is the oracle sharded
    by (b, h).  Returns (tokens/s, cores)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            times = pool.map_async(_oracle_shard, [w.name] * n).get(timeout=600)
    except (mp.TimeoutError, OSError):
        return None, n
    return n * oracle_tokens_per_s(w, w.N, 1.0) / max(times), n


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def run_reference(args, w, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    sample = cpu_slice(w)
    rows = sample_rows(w)
    for _ in range(args.warmup):
        oracle_step(w, sample, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, sample, rows)
    dt = (time.perf_counter() - t0) / args.steps
    val = oracle_tokens_per_s(w, len(rows), dt)
    n = w.N // w.C
    desc = (f"per step the queries of chunks {n // 4} and {3 * n // 4 - 1} ({len(rows)} queries) "
            f"of one full-length (N={w.N}) slice of {w.name}: encode, select, attend fwd + bwd; "
            "tokens/s = queries / H / time")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_K": w.d_K,
                   "d_V": w.d_V, "k": w.k, "C": w.C, "bits": w.bits},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- our arm ---

def launches_per_step(w, fwd_only=False) -> int:
    """Kernel launches the library makes for one step (encode x2, sort, select,
    attend fwd, attend bwd), following its launch structure."""
    n = w.N // w.C
    code_passes = max(1, -(-(w.d_K * w.bits) // 8))
    sort = 3 * code_passes + 3 if n >= 2 else 0
    fwd = 2 + sort + 1 + 1
    if fwd_only:
        return fwd
    key_bits = max(1, int(np.ceil(np.log2(max(w.N, 2)))))
    idx_passes = max(1, -(-key_bits // 8))
    bwd = 1 + 3 * idx_passes + 1 + 1 + 2
    return fwd + bwd


def run_ours(args, w, rank, world):
    import torch
    import torch.distributed as dist

    from order_retrieval_gb300 import binding as zb
    from order_retrieval_gb300 import workloads as W
    from order_retrieval_gb300.pipeline import ZetaPlan

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wr = w.replace(seed=w.seed + 1000 * rank)          # every rank its own batch
    g = W.generate(wr, with_dout=True)
    p = zb.problem_of(wr)
    warm = max(3, args.warmup)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak_mb = {}

    def mem_start():
        """Peak-memory window of one workload: everything it allocates from
        here on (inputs, buffers, workspaces) is counted."""
        torch.cuda.synchronize(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        return torch.cuda.memory_allocated(dev)

    def mem_peak(base):
        torch.cuda.synchronize(dev)
        return (torch.cuda.max_memory_allocated(dev) - base) / 2 ** 20

    mem0 = mem_start()

    def to_dev(a, vals=False):
        t = torch.from_numpy(np.ascontiguousarray(a)).reshape(-1)
        if vals and a.dtype == np.int16:
            t = t.view(torch.bfloat16)
        return t.pin_memory(), t.to(dev)

    (q_h, q), (k_h, k), (v_h, v), (g_h, gamma), (do_h, dout) = (
        to_dev(g["q"]), to_dev(g["k"]), to_dev(g["v"], True), to_dev(g["gamma"]),
        to_dev(g["dout"], True))
    plan = ZetaPlan(p, dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # --- the step as one CUDA graph: encode x2, sort, select, attend fwd, attend bwd
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warm):
            plan.forward(q, k, v, gamma)
            plan.backward(q, k, v, gamma, dout)
    torch.cuda.current_stream().wait_stream(side)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        plan.forward(q, k, v, gamma)
        plan.backward(q, k, v, gamma, dout)
    fwd_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fwd_graph):
        plan.forward(q, k, v, gamma)
    for _ in range(warm):
        step_graph.replay()
        if world > 1:
            dist.all_reduce(plan.dgamma)
        flush.zero_()
    barrier()
    if int(plan.status.item()) != 0:
        raise RuntimeError(f"device status {plan.status.item()}")
    peak_mb[w.name + " (fwd+bwd)"] = mem_peak(mem0)

    # --- timed: K graph replays, each bracketed by events; L2 flushed between steps
    step_ms = []
    with ClockSampler(physical_gpu_index(dev.index or 0)) as clk:
        barrier()
        t_wall = time.perf_counter()
        for _ in range(args.steps):
            a, b = ev(), ev()
            a.record()
            step_graph.replay()
            if world > 1:
                dist.all_reduce(plan.dgamma)
            b.record()
            flush.zero_()
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
        barrier()
        wall = time.perf_counter() - t_wall
    dev_ms = sum(step_ms) / len(step_ms)
    step_stats = {"mean": dev_ms, "median": statistics.median(step_ms), "min": min(step_ms),
                  "max": max(step_ms), "n": len(step_ms)}
    t = torch.tensor([dev_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dev_ms = float(t.item())
    tokens = wr.B * wr.N * world
    value = tokens / (dev_ms * 1e-3)

    # --- forward alone (graph), and a per-call breakdown of the step (direct calls)
    fwd_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record()
        fwd_graph.replay()
        b.record()
        b.synchronize()
        fwd_ms.append(a.elapsed_time(b))
    fwd_train_ms = sum(fwd_ms) / len(fwd_ms)
    calls = ["encode", "sort", "select", "attend_fwd", "attend_bwd"]
    per_call = {c: 0.0 for c in calls}
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(6)]
        e[0].record()
        zb.zeta_encode(p, q, plan.q_codes)
        zb.zeta_encode(p, k, plan.k_codes)
        e[1].record()
        zb.zeta_sort_chunks(p, plan.k_codes, plan.prefix_codes, plan.prefix_idx, plan.sort_ws)
        e[2].record()
        zb.zeta_select_topk(p, plan.q_codes, plan.prefix_codes, plan.prefix_idx, plan.idx)
        e[3].record()
        zb.zeta_attend_fwd(p, q, k, v, gamma, plan.idx, plan.out, plan.rowsum, plan.status)
        e[4].record()
        zb.zeta_attend_bwd(p, q, k, v, gamma, plan.idx, dout, plan.dq, plan.dk, plan.dv,
                           plan.dgamma, plan.bwd_ws, plan.status)
        e[5].record()
        e[5].synchronize()
        for c, (x, y) in zip(calls, zip(e[:-1], e[1:])):
            per_call[c] += x.elapsed_time(y) / args.steps

    # --- end to end through the C ABI with host buffers (pinned): every step
    # copies its inputs host -> device, runs the five calls, and copies its
    # results device -> host.  Serial: one stream, step after step.  Pipelined
    # (the e2e figure): NSETS device buffer sets; step n+1's inputs go up on a
    # copy stream while step n computes, and step n's results come down on
    # another while step n+1 computes, a set being reused only after its
    # previous results are down; each set's five calls are replayed as one
    # CUDA graph.  Both time every copy of every step.
    NSETS = 3
    out_h = [torch.empty(plan.out.numel(), dtype=plan.out.dtype).pin_memory()
             for _ in range(NSETS)]
    dq_h = [torch.empty(plan.dq.numel(), dtype=torch.float32).pin_memory() for _ in range(NSETS)]
    dk_h = [torch.empty(plan.dk.numel(), dtype=torch.float32).pin_memory() for _ in range(NSETS)]
    dv_h = [torch.empty(plan.dv.numel(), dtype=plan.dv.dtype).pin_memory() for _ in range(NSETS)]
    dg_h = [torch.empty(plan.dgamma.numel(), dtype=torch.float32).pin_memory()
            for _ in range(NSETS)]
    ins_h = (q_h, k_h, v_h, g_h, do_h)
    h2d = sum(x.numel() * x.element_size() for x in ins_h)
    d2h = sum(x[0].numel() * x[0].element_size() for x in (out_h, dq_h, dk_h, dv_h, dg_h))

    def outs(pl):
        return (pl.out, pl.dq, pl.dk, pl.dv, pl.dgamma)

    def hosts(bi):
        return (out_h[bi], dq_h[bi], dk_h[bi], dv_h[bi], dg_h[bi])

    e2e_ms = []
    for it in range(warm + args.steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record()
        for src, dst in zip(ins_h, (q, k, v, gamma, dout)):
            dst.copy_(src, non_blocking=True)
        plan.forward(q, k, v, gamma)
        plan.backward(q, k, v, gamma, dout)
        if world > 1:
            dist.all_reduce(plan.dgamma)
        for src, dst in zip(outs(plan), hosts(0)):
            dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        if it >= warm:
            e2e_ms.append(a.elapsed_time(b))
    e2e_serial = tokens / (sum(e2e_ms) / len(e2e_ms) * 1e-3)

    plans = [plan] + [ZetaPlan(p, dev) for _ in range(NSETS - 1)]
    dev_in = [(q, k, v, gamma, dout)] + [tuple(t.clone() for t in (q, k, v, gamma, dout))
                                         for _ in range(NSETS - 1)]
    # each set's five calls as one CUDA graph, as in the timed step (one eager
    # pass of every set first)
    for bi in range(1, NSETS):
        plans[bi].forward(*dev_in[bi][:4])
        plans[bi].backward(*dev_in[bi])
    torch.cuda.synchronize()
    comp_graphs = []
    for bi in range(NSETS):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            plans[bi].forward(*dev_in[bi][:4])
            plans[bi].backward(*dev_in[bi])
        comp_graphs.append(g_)
    # compute on a stream of its own: on the legacy default stream the steps'
    # kernels would serialise with the copies on the other streams
    comp = torch.cuda.Stream(dev)
    cp_in, cp_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done = [ev() for _ in range(NSETS)]
    out_done = [ev() for _ in range(NSETS)]
    in_ready = [ev() for _ in range(NSETS)]
    started = [False] * NSETS

    def pipelined_steps(n, stages=None):
        # stages: if given, gets per step the start events of its H2D copies,
        # compute and D2H copies (their ends are in_ready, comp_done, out_done)
        for it in range(n):
            bi = it % NSETS
            st3 = [ev(), ev(), ev()] if stages is not None else None
            with torch.cuda.stream(cp_in):
                if started[bi]:
                    cp_in.wait_event(comp_done[bi])       # the set's previous step computed
                if st3:
                    st3[0].record(cp_in)
                for src, dst in zip(ins_h, dev_in[bi]):
                    dst.copy_(src, non_blocking=True)
                in_ready[bi].record(cp_in)
            comp.wait_event(in_ready[bi])
            if started[bi]:
                comp.wait_event(out_done[bi])             # and its results copied out
            with torch.cuda.stream(comp):
                if st3:
                    st3[1].record(comp)
                comp_graphs[bi].replay()
                if world > 1:
                    dist.all_reduce(plans[bi].dgamma)
                comp_done[bi].record(comp)
            with torch.cuda.stream(cp_out):
                cp_out.wait_event(comp_done[bi])
                if st3:
                    st3[2].record(cp_out)
                for src, dst in zip(outs(plans[bi]), hosts(bi)):
                    dst.copy_(src, non_blocking=True)
                out_done[bi].record(cp_out)
            started[bi] = True
            if st3:
                # the end events are reused by later steps: time them now, on
                # copies of this step's ends
                ends = [ev(), ev(), ev()]
                ends[0].record(cp_in)
                ends[1].record(comp)
                ends[2].record(cp_out)
                stages.append((st3, ends))

    # five timed trials of K steps each, the median reported: the host copies
    # share the machine's host memory and links with other jobs, which moves
    # single trials by up to 20 %
    pipelined_steps(warm)
    torch.cuda.synchronize()
    barrier()
    e2e_trials, e2e_host_ms, e2e_stage_ms = [], [], []
    for _ in range(5):
        t_a = ev()
        t_a.record(cp_in)
        h0 = time.perf_counter()
        stages = []
        pipelined_steps(args.steps, stages)
        t_b = ev()
        t_b.record(cp_out)
        e2e_host_ms.append((time.perf_counter() - h0) * 1e3)     # host enqueue of the trial
        t_b.synchronize()
        torch.cuda.synchronize()
        # mean H2D, compute and D2H time per step of the trial
        e2e_stage_ms.append([statistics.mean(st[i].elapsed_time(en[i]) for st, en in stages)
                             for i in range(3)])
        tt = torch.tensor([t_a.elapsed_time(t_b)], dtype=torch.float64, device=dev)
        if world > 1:
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_trials.append(tokens * args.steps / (float(tt.item()) * 1e-3))
        barrier()
    e2e = statistics.median(e2e_trials)
    del comp_graphs, plans, dev_in

    # --- efficiency workload: forward alone, and the attend-forward kernel roofline
    we = W.EFFICIENCY.replace(seed=W.EFFICIENCY.seed + 1000 * rank)
    ge = W.generate(we)
    pe = zb.problem_of(we)
    mem_e = mem_start()
    qe, ke = to_dev(ge["q"])[1], to_dev(ge["k"])[1]
    ve, gme = to_dev(ge["v"], True)[1], to_dev(ge["gamma"])[1]
    plan_e = ZetaPlan(pe, dev, backward=False)
    for _ in range(warm):
        plan_e.forward(qe, ke, ve, gme)
    peak_mb[we.name + " (fwd)"] = mem_peak(mem_e)
    fwd_e, att_e = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(3)]
        e[0].record()
        zb.zeta_encode(pe, qe, plan_e.q_codes)
        zb.zeta_encode(pe, ke, plan_e.k_codes)
        zb.zeta_sort_chunks(pe, plan_e.k_codes, plan_e.prefix_codes, plan_e.prefix_idx,
                            plan_e.sort_ws)
        zb.zeta_select_topk(pe, plan_e.q_codes, plan_e.prefix_codes, plan_e.prefix_idx,
                            plan_e.idx)
        e[1].record()
        zb.zeta_attend_fwd(pe, qe, ke, ve, gme, plan_e.idx, plan_e.out, plan_e.rowsum,
                           plan_e.status)
        e[2].record()
        e[2].synchronize()
        fwd_e.append(e[0].elapsed_time(e[2]))
        att_e.append(e[1].elapsed_time(e[2]))
    fwd_e_ms = sum(fwd_e) / len(fwd_e)
    att_e_ms = sum(att_e) / len(att_e)
    warm_e = []                               # the same launch with a warm L2
    for _ in range(args.steps):
        e = [ev() for _ in range(2)]
        e[0].record()
        zb.zeta_attend_fwd(pe, qe, ke, ve, gme, plan_e.idx, plan_e.out, plan_e.rowsum,
                           plan_e.status)
        e[1].record()
        e[1].synchronize()
        warm_e.append(e[0].elapsed_time(e[1]))
    att_warm_ms = sum(warm_e) / len(warm_e)

    # --- fused select + attend (one launch) on the same workload
    plan_f = ZetaPlan(pe, dev, backward=False, fused=True)
    for _ in range(warm):
        plan_f.forward(qe, ke, ve, gme)
    fus_tot, fus_k = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(3)]
        e[0].record()
        zb.zeta_encode(pe, qe, plan_f.q_codes)
        zb.zeta_encode(pe, ke, plan_f.k_codes)
        zb.zeta_sort_chunks(pe, plan_f.k_codes, plan_f.prefix_codes, plan_f.prefix_idx,
                            plan_f.sort_ws)
        e[1].record()
        zb.zeta_select_attend_fwd(pe, qe, ke, ve, gme, plan_f.q_codes, plan_f.prefix_codes,
                                  plan_f.prefix_idx, plan_f.idx, plan_f.out, plan_f.rowsum,
                                  plan_f.status)
        e[2].record()
        e[2].synchronize()
        fus_tot.append(e[0].elapsed_time(e[2]))
        fus_k.append(e[1].elapsed_time(e[2]))
    if int(plan_f.status.item()) != 0:
        raise RuntimeError(f"device status {plan_f.status.item()} (fused)")
    fus_tot_ms = sum(fus_tot) / len(fus_tot)
    fus_k_ms = sum(fus_k) / len(fus_k)
    del plan_f

    # --- the 1,048,576-token workload (B=1, H=8, k=64, C=4096): forward alone,
    # its index part (encode, sort, select) and the attend kernel
    wl = W.LONG.replace(seed=W.LONG.seed + 1000 * rank)
    gl = W.generate(wl)
    pl = zb.problem_of(wl)
    mem_l = mem_start()
    ql, kl = to_dev(gl["q"])[1], to_dev(gl["k"])[1]
    vl, gml = to_dev(gl["v"], True)[1], to_dev(gl["gamma"])[1]
    del gl
    plan_l = ZetaPlan(pl, dev, backward=False)
    for _ in range(warm):
        plan_l.forward(ql, kl, vl, gml)
    peak_mb[wl.name + " (fwd)"] = mem_peak(mem_l)
    long_tot, long_idx = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(3)]
        e[0].record()
        zb.zeta_encode(pl, ql, plan_l.q_codes)
        zb.zeta_encode(pl, kl, plan_l.k_codes)
        zb.zeta_sort_chunks(pl, plan_l.k_codes, plan_l.prefix_codes, plan_l.prefix_idx,
                            plan_l.sort_ws)
        zb.zeta_select_topk(pl, plan_l.q_codes, plan_l.prefix_codes, plan_l.prefix_idx,
                            plan_l.idx)
        e[1].record()
        zb.zeta_attend_fwd(pl, ql, kl, vl, gml, plan_l.idx, plan_l.out, plan_l.rowsum,
                           plan_l.status)
        e[2].record()
        e[2].synchronize()
        long_tot.append(e[0].elapsed_time(e[2]))
        long_idx.append(e[0].elapsed_time(e[1]))
    if int(plan_l.status.item()) != 0:
        raise RuntimeError(f"device status {plan_l.status.item()} (1M tokens)")
    long_ms = sum(long_tot) / len(long_tot)
    long_idx_ms = sum(long_idx) / len(long_idx)
    del plan_l, ql, kl, vl, gml
    torch.cuda.empty_cache()

    variants = {}
    # --- the pages' 12-bit grid (36-bit codes in 64-bit words) on the same
    # workload: the whole forward, and its index part
    w12 = we.replace(bits=12)
    p12 = zb.problem_of(w12)
    plan12 = ZetaPlan(p12, dev, backward=False)
    for _ in range(warm):
        plan12.forward(qe, ke, ve, gme)
    tot12, idx12 = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(3)]
        e[0].record()
        zb.zeta_encode(p12, qe, plan12.q_codes)
        zb.zeta_encode(p12, ke, plan12.k_codes)
        zb.zeta_sort_chunks(p12, plan12.k_codes, plan12.prefix_codes, plan12.prefix_idx,
                            plan12.sort_ws)
        zb.zeta_select_topk(p12, plan12.q_codes, plan12.prefix_codes, plan12.prefix_idx,
                            plan12.idx)
        e[1].record()
        zb.zeta_attend_fwd(p12, qe, ke, ve, gme, plan12.idx, plan12.out, plan12.rowsum,
                           plan12.status)
        e[2].record()
        e[2].synchronize()
        tot12.append(e[0].elapsed_time(e[2]))
        idx12.append(e[0].elapsed_time(e[1]))
    if int(plan12.status.item()) != 0:
        raise RuntimeError(f"device status {plan12.status.item()} (12-bit grid)")
    ms12 = sum(tot12) / len(tot12)
    variants["grid12"] = {"workload": we.name + " with bits=12 (u64 codes)",
                          "fwd_tokens_per_s": we.B * we.N * world / (ms12 * 1e-3),
                          "fwd_ms": ms12, "encode_sort_select_ms": sum(idx12) / len(idx12)}
    del plan12

    # --- multi-curve variant (3 cyclic / 6 permuted coordinate orders) on the
    # efficiency workload: the whole forward, and its index part
    for curves in (3, 6):
        pc = ZetaPlan(pe, dev, backward=False, curves=curves)
        for _ in range(warm):
            pc.forward(qe, ke, ve, gme)
        tot, sel = [], []
        for _ in range(args.steps):
            flush.zero_()
            e = [ev() for _ in range(3)]
            e[0].record()
            zb.zeta_encode_curves(pe, qe, pc.axes, pc.q_codes)
            zb.zeta_encode_curves(pe, ke, pc.axes, pc.k_codes)
            zb.zeta_sort_chunks(pc.p_sort, pc.k_codes, pc.prefix_codes, pc.prefix_idx,
                                pc.sort_ws)
            zb.zeta_select_topk_curves(pe, curves, pc.q_codes, pc.prefix_codes, pc.prefix_idx,
                                       pc.idx)
            e[1].record()
            zb.zeta_attend_fwd(pe, qe, ke, ve, gme, pc.idx, pc.out, pc.rowsum, pc.status)
            e[2].record()
            e[2].synchronize()
            tot.append(e[0].elapsed_time(e[2]))
            sel.append(e[0].elapsed_time(e[1]))
        if int(pc.status.item()) != 0:
            raise RuntimeError(f"device status {pc.status.item()} ({curves} curves)")
        ms = sum(tot) / len(tot)
        variants[f"curves{curves}"] = {
            "workload": we.name, "fwd_tokens_per_s": we.B * we.N * world / (ms * 1e-3),
            "fwd_ms": ms, "encode_sort_select_ms": sum(sel) / len(sel)}
        del pc

    # --- projection front end fused with the encode (tcgen05), the training
    # workload's tokens with D = 512 features: the kernel alone, then the whole
    # forward from features (project, sort, select, attend)
    pj = W.PROJ
    gp = W.generate_projection(pj)
    pp = zb.problem_of(pj.base)

    def bf16_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).reshape(-1).to(dev)

    xp, w1p = bf16_dev(gp["x"]), bf16_dev(gp["W1"])
    b1p, w2p, b2p = (torch.from_numpy(gp[n]).reshape(-1).to(dev) for n in ("b1", "W2", "b2"))
    plan_p = ZetaPlan(pp, dev, backward=False)
    qp = torch.empty(pp.B * pp.H * pp.N * pp.d_K, dtype=torch.float32, device=dev)
    kp = torch.empty_like(qp)

    def project():
        zb.zeta_project_encode(pp, pj.D, pj.F, xp, w1p, b1p, w2p, b2p, qp, kp, plan_p.q_codes,
                               plan_p.k_codes, plan_p.status)

    for _ in range(warm):
        project()
    pr_ms, pf_ms = [], []
    for _ in range(args.steps):
        flush.zero_()
        e = [ev() for _ in range(3)]
        e[0].record()
        project()
        e[1].record()
        zb.zeta_sort_chunks(pp, plan_p.k_codes, plan_p.prefix_codes, plan_p.prefix_idx,
                            plan_p.sort_ws)
        zb.zeta_select_topk(pp, plan_p.q_codes, plan_p.prefix_codes, plan_p.prefix_idx,
                            plan_p.idx)
        zb.zeta_attend_fwd(pp, qp, kp, v, gamma, plan_p.idx, plan_p.out, plan_p.rowsum,
                           plan_p.status)
        e[2].record()
        e[2].synchronize()
        pr_ms.append(e[0].elapsed_time(e[1]))
        pf_ms.append(e[0].elapsed_time(e[2]))
    if int(plan_p.status.item()) != 0:
        raise RuntimeError(f"device status {plan_p.status.item()} (projection)")
    proj_ms = sum(pr_ms) / len(pr_ms)
    proj_flop = 2.0 * pp.B * pp.N * pj.D * (2 * pp.H * pj.F)
    variants["projection"] = {
        "workload": pj.name, "kernel_ms": proj_ms, "tflops": proj_flop / (proj_ms * 1e-3) / 1e12,
        "fwd_from_features_tokens_per_s": tokens / (sum(pf_ms) / len(pf_ms) * 1e-3),
        "fwd_from_features_ms": sum(pf_ms) / len(pf_ms)}
    del plan_p

    # --- alternative weight kernels (softmax of -d2/gamma^2, inverse Euclidean)
    # on the timed workload: the whole step, captured and timed like the main one
    for weight in ("softmax", "inv_euclid"):
        pw = zb.problem_of(wr, weight=weight)
        pln = ZetaPlan(pw, dev)
        with torch.cuda.stream(side):
            for _ in range(warm):
                pln.forward(q, k, v, gamma)
                pln.backward(q, k, v, gamma, dout)
        torch.cuda.current_stream().wait_stream(side)
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            pln.forward(q, k, v, gamma)
            pln.backward(q, k, v, gamma, dout)
        fgph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgph):
            pln.forward(q, k, v, gamma)
        tms, fms = [], []
        for it in range(warm + args.steps):
            for gr, lst in ((gph, tms), (fgph, fms)):
                flush.zero_()
                a, b = ev(), ev()
                a.record()
                gr.replay()
                b.record()
                b.synchronize()
                if it >= warm:
                    lst.append(a.elapsed_time(b))
        if int(pln.status.item()) != 0:
            raise RuntimeError(f"device status {pln.status.item()} ({weight})")
        sms, fmean = sum(tms) / len(tms), sum(fms) / len(fms)
        variants[weight] = {"workload": wr.name, "tokens_per_s": tokens / (sms * 1e-3),
                            "ms_per_step": sms, "fwd_tokens_per_s": tokens / (fmean * 1e-3),
                            "fwd_ms": fmean}
        del pln, gph, fgph

    if rank != 0:
        return
    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    fb = fwd_attend_bytes(we)
    achieved = fb / (att_e_ms * 1e-3) / 1e9
    fbt = fwd_attend_bytes(wr)
    bb = bwd_attend_bytes(wr)

    # CPU baseline: the oracle on one full-length slice of this workload
    import oracle
    oracle.build()
    sample = cpu_slice(w)
    t0 = time.perf_counter()
    oracle_step(w, sample)
    cpu_dt = time.perf_counter() - t0
    sharded_rate, sharded_cores = cpu_sharded(w)
    digest = sources_digest(ATTEND_FWD_SOURCES)
    traffic = (ATTEND_FWD_TRAFFIC["bytes"]
               if ATTEND_FWD_TRAFFIC["sources_sha256"] == digest else None)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": dev_ms,
        "ms_per_step_stats": step_stats,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "v, dO, out, dv bf16; q, k, weights and accumulation f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_K": w.d_K,
                   "d_V": w.d_V, "k": w.k, "C": w.C, "bits": w.bits,
                   "l2": "flushed between steps (256 MiB write); inputs larger than L2",
                   "step": "one CUDA graph: encode q,k; sort; select; attend fwd; attend bwd",
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "fwd_tokens_per_s": tokens / (fwd_train_ms * 1e-3),
        "fwd_efficiency": {"workload": we.name, "tokens_per_s": we.B * we.N * world /
                           (fwd_e_ms * 1e-3), "ms": fwd_e_ms, "attend_fwd_ms": att_e_ms,
                           "attend_fwd_ms_warm_l2": att_warm_ms},
        "fwd_long": {"workload": wl.name, "tokens_per_s": wl.B * wl.N * world / (long_ms * 1e-3),
                     "ms": long_ms, "encode_sort_select_ms": long_idx_ms,
                     "attend_fwd_ms": long_ms - long_idx_ms,
                     "attend_fwd_frac": fwd_attend_bytes(wl) / ((long_ms - long_idx_ms) * 1e-3)
                                        / 1e9 / hbm_peak},
        "peak_device_mb": {**peak_mb, "how": "torch max_memory_allocated over each workload's "
                                              "inputs, buffers, workspaces and outputs (the "
                                              "library allocates nothing itself)",
                           "pages_fwd_65536_tokens_mb": PAGES_FWD_MB},
        "fwd_efficiency_fused": {
            "workload": we.name, "call": "zeta_select_attend_fwd",
            "tokens_per_s": we.B * we.N * world / (fus_tot_ms * 1e-3), "ms": fus_tot_ms,
            "select_attend_ms": fus_k_ms,
            "roofline": {"bound": "hbm", "achieved": fused_fwd_bytes(we) / (fus_k_ms * 1e-3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": fused_fwd_bytes(we) / (fus_k_ms * 1e-3) / 1e9 / hbm_peak,
                         "algorithmic_bytes": fused_fwd_bytes(we)}},
        "per_call_ms": per_call,
        "variants": variants,
        "roofline": {"kernel": "attend_fwd_tc (efficiency workload, L2 flushed)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "traffic_source": ATTEND_FWD_TRAFFIC["capture"] + (
                         "" if traffic is not None else " (null: kernel sources changed since)"),
                     "algorithmic_bytes": fb, "peak_source": peak_src},
        "roofline_projection": {
            "kernel": "project_encode_tc (tcgen05, B=4 N=65536 D=512 F=64, L2 flushed)",
            "bound": "tensor", "achieved": variants["projection"]["tflops"],
            "peak": peaks.get("bf16_tflops", 1900.0), "unit": "TFLOP/s",
            "frac": variants["projection"]["tflops"] / peaks.get("bf16_tflops", 1900.0),
            "peak_source": "measured (cuBLAS bf16 burst)" if "bf16_tflops" in peaks
                           else "fallback"},
        "roofline_train": {
            "attend_fwd": {"achieved": fbt / (per_call["attend_fwd"] * 1e-3) / 1e9,
                           "frac": fbt / (per_call["attend_fwd"] * 1e-3) / 1e9 / hbm_peak,
                           "algorithmic_bytes": fbt},
            "attend_bwd": {"achieved": bb / (per_call["attend_bwd"] * 1e-3) / 1e9,
                           "frac": bb / (per_call["attend_bwd"] * 1e-3) / 1e9 / hbm_peak,
                           "algorithmic_bytes": bb},
            "unit": "GB/s"},
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "pinned host buffers; per step H2D of q, k, v, gamma, dO, the five calls "
                       "(one CUDA graph per buffer set), D2H of out, dq, dk, dv, dgamma; three "
                       "buffer sets, copies on side "
                       "streams overlapping the neighbouring steps' compute on a third; median "
                       "of five trials of K steps",
                "trials": e2e_trials,
                "trial_host_enqueue_ms": e2e_host_ms,
                "trial_step_h2d_compute_d2h_ms": e2e_stage_ms,
                "serial_value": e2e_serial},
        "gpu_launches": launches_per_step(w) * args.steps,
        "cpu_baseline": {"value": oracle_tokens_per_s(w, w.N, cpu_dt), "unit": "tokens/s",
                         "cores": 1, "kind": "oracle",
                         "sample": f"one full-length slice (N={w.N} queries of one head) of "
                                   f"{w.name}: encode, select, attend fwd + bwd; extrapolated "
                                   f"to the B*H = {w.B * w.H} slices of a step "
                                   "(tokens/s = N / H / time of the slice)",
                         "slice_s": cpu_dt,
                         "cpu_model": cpu_model(),
                         "sharded": {"value": sharded_rate, "unit": "tokens/s",
                                     "cores": sharded_cores,
                                     "how": "one spawned process per host core, each on "
                                            "a full slice (slices are independent)"}},
        "clocks": clk.summary(),
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    args = ap.parse_args()
    from order_retrieval_gb300 import workloads as W
    w = W.TRAIN
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
