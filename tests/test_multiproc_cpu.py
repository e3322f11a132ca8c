"""World-size-2 CPU test of the multi-GPU arrangement (gloo backend).

The path shards over (b, h): each rank owns a batch slice and computes its
own outputs; the only exchange is the gamma gradient, a sum over b that
becomes an all-reduce across ranks.  Here each rank runs the CPU oracle on
its half of the batch and the all-reduced dgamma must equal the oracle's
dgamma over the whole batch."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _slice_grads(w, g, b, h):
    import oracle
    from order_retrieval_gb300 import workloads as W
    q, k = g["q"][b, h], g["k"][b, h]
    v = W.values_f64(w, g["v"][b, h])
    do = W.values_f64(w, g["dout"][b, h])
    qc, kc = oracle.encode(q, w.bits), oracle.encode(k, w.bits)
    idx = oracle.select(qc[None], kc[None], w.C, w.k)[0]
    return oracle.attend_bwd(q, k, v, float(g["gamma"][h]), idx, do, w.C)


def _worker(rank, world, port, out_path):
    import sys
    sys.path.insert(0, ROOT)
    from order_retrieval_gb300 import workloads as W
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.TINY.replace(B=4, H=2, N=256, C=64, k=8)
    g = W.generate(w, with_dout=True)
    dg = torch.zeros(w.H, dtype=torch.float64)
    for b in range(rank, w.B, world):           # this rank's share of the batch
        for h in range(w.H):
            dg[h] += _slice_grads(w, g, b, h)[3]
    dist.all_reduce(dg)
    if rank == 0:
        np.save(out_path, dg.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_dgamma_allreduce_over_batch_shards(tmp_path):
    from order_retrieval_gb300 import workloads as W
    out = str(tmp_path / "dg.npy")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True,
                       start_method="spawn")
    w = W.TINY.replace(B=4, H=2, N=256, C=64, k=8)
    g = W.generate(w, with_dout=True)
    ref = np.zeros(w.H)
    for b in range(w.B):
        for h in range(w.H):
            ref[h] += _slice_grads(w, g, b, h)[3]
    np.testing.assert_allclose(np.load(out), ref, rtol=1e-12, atol=1e-12)
