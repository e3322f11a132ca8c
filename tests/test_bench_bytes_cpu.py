"""The bench's algorithmic-byte models, pinned to per-unit counts worked out by
hand.  Every roofline fraction the bench prints divides these bytes by a
measured time, so a wrong term here would move every reported fraction.

Per query-head (bf16 values, d_V = 64, d_K = 3, 4-byte indices and floats):
- attend forward, k = 64: each of the k window keys brings a value row
  (128 B), its coordinates (12 B) and its index (4 B) = 144 B; the query's own
  q (12 B), output row (128 B) and row sum (4 B) = 144 B; its key's own-chunk
  k and v rows once (140 B).  64 * 144 + 144 + 140 = 9,500 B.
- fused select + attend adds the query's code (4 B), one 4-byte code per
  halving of the largest prefix (N - C = 64,512 keys: 16 probes, 64 B) and the
  index row written back (64 * 4 = 256 B): 9,500 + 324 = 9,824 B.
- attend backward, k = 48: per window key a value row on the query side and a
  dO row on the key side (2 * 128 B), coordinates twice (2 * 12 B) and four
  index words (idx read twice, the transpose written and read: 16 B) = 296 B;
  per query dO (128 B), q and dq (24 B) and 16 B of scalars handed to the key
  side = 168 B; per key its own-chunk k, v and dO rows (3 * 140 B) and dk, dv
  (140 B) = 560 B.
  48 * 296 + 168 + 560 = 14,936 B.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from order_retrieval_gb300 import workloads as W  # noqa: E402


def _query_heads(w):
    return w.B * w.H * w.N


def test_forward_bytes_efficiency_workload():
    w = W.EFFICIENCY
    assert (w.k, w.d_V, w.d_K, w.v_dtype) == (64, 64, 3, "bf16")
    assert _query_heads(w) == 524_288
    assert bench.fwd_attend_bytes(w) == 9_500 * 524_288 == 4_980_736_000


def test_fused_bytes_efficiency_workload():
    w = W.EFFICIENCY
    assert w.d_K * w.bits <= 32                       # 4-byte codes
    assert (w.N - w.C) == 64_512 and (w.N - w.C).bit_length() == 16
    assert bench.fused_fwd_bytes(w) == 9_824 * 524_288


def test_backward_bytes_training_workload():
    w = W.TRAIN
    assert (w.k, w.d_V, w.d_K, w.v_dtype) == (48, 64, 3, "bf16")
    assert _query_heads(w) == 2_097_152
    assert bench.bwd_attend_bytes(w) == 14_936 * 2_097_152 == 31_323_062_272


def test_forward_bytes_training_workload():
    # k = 48: 48 * 144 + 144 + 140 = 7,196 B per query-head
    w = W.TRAIN
    assert bench.fwd_attend_bytes(w) == 7_196 * 2_097_152


def test_f32_values_double_the_value_bytes():
    # f32 values: a value row is 256 B, so 64 * (256 + 16) + 12 + 256 + 4 + 12 + 256
    w = W.EFFICIENCY.replace(v_dtype="f32")
    assert bench.fwd_attend_bytes(w) == (64 * 272 + 540) * 524_288
