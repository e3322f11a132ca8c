"""Seeded synthetic workloads for the ZETA hot path.

This module holds only input generation: problem sizes and seeded random draws.
It contains none of the method's arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), written here with numpy uint64
arithmetic so the draws are bit-identical on every host.  Uniforms on [-1, 1)
take the top 24 bits of a draw (exact in float32); Gaussians use the Box-Muller
transform in double precision.  bf16 values are produced by round-to-nearest-even
from float32 and are carried as their 16-bit patterns (numpy int16).

Each workload draws its tensors from one stream, in the order q, k, v, gamma,
dO, so that a given seed always yields the same tensors.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

_PHI = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22


class SplitMix64:
    """Counter-form SplitMix64: draw i is mix(seed + (i + 1) * phi)."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed)
        self.pos = 0

    def raw(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint64)
        with np.errstate(over="ignore"):
            for s in range(0, n, _BLOCK):
                m = min(_BLOCK, n - s)
                ctr = np.arange(self.pos + s + 1, self.pos + s + 1 + m, dtype=np.uint64)
                z = self.seed + ctr * _PHI
                z = (z ^ (z >> np.uint64(30))) * _M1
                z = (z ^ (z >> np.uint64(27))) * _M2
                out[s:s + m] = z ^ (z >> np.uint64(31))
        self.pos += n
        return out

    def uniform_pm1_f32(self, n: int) -> np.ndarray:
        """Float32 uniform on [-1, 1) on the 2^-23 grid (exact)."""
        out = np.empty(n, dtype=np.float32)
        for s in range(0, n, _BLOCK):
            m = min(_BLOCK, n - s)
            top = (self.raw(m) >> np.uint64(40)).astype(np.int64) - (1 << 23)
            out[s:s + m] = top.astype(np.float32) * np.float32(2.0 ** -23)
        return out

    def uniform01_f64(self, n: int) -> np.ndarray:
        """Double uniform on [0, 1) with 53 random bits."""
        return (self.raw(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def normal_f64(self, n: int) -> np.ndarray:
        """Standard normal draws by Box-Muller (two uniforms per pair)."""
        out = np.empty(n, dtype=np.float64)
        for s in range(0, n, _BLOCK):
            m = min(_BLOCK, n - s)
            pairs = (m + 1) // 2
            u = self.uniform01_f64(2 * pairs).reshape(pairs, 2)
            rad = np.sqrt(-2.0 * np.log1p(-u[:, 0]))        # 1 - u in (0, 1]
            ang = 2.0 * np.pi * u[:, 1]
            z = np.empty((pairs, 2), dtype=np.float64)
            z[:, 0] = rad * np.cos(ang)
            z[:, 1] = rad * np.sin(ang)
            out[s:s + m] = z.reshape(-1)[:m]
        return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even); returns the bit patterns as int16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    r = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r.view(np.int16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (int16/uint16) to float32 exactly."""
    u = np.ascontiguousarray(b).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One problem instance of the ZETA hot path.

    B batch, H heads, N tokens, d_K query/key width, d_V value width, k window
    size, C chunk length, bits grid bits per coordinate, v_dtype 'f32' or 'bf16',
    gamma: a float (every head) or (lo, hi) for per-head uniform draws,
    dist: 'uniform' (U[-1,1)) or 'clusters' (64-Gaussian mixture), v_dist:
    'uniform' or 'normal'."""
    name: str
    B: int
    H: int
    N: int
    d_K: int
    d_V: int
    k: int
    C: int
    bits: int
    v_dtype: str
    gamma: object
    dist: str
    v_dist: str
    seed: int

    @property
    def n_chunks(self) -> int:
        return self.N // self.C

    @property
    def prefix_entries(self) -> int:
        n = self.n_chunks
        return self.C * n * (n - 1) // 2

    @property
    def code_bits(self) -> int:
        return self.d_K * self.bits

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five problem instances used for parity and timing.
TINY = Workload("tiny_f32_n1024", 1, 1, 1024, 3, 32, 32, 128, 10, "f32", 0.5,
                "uniform", "uniform", 0)
CLUSTERED = Workload("clustered_bf16_n4096", 2, 8, 4096, 3, 64, 32, 256, 10, "bf16",
                     (0.3, 1.0), "clusters", "normal", 1)
EFFICIENCY = Workload("efficiency_bf16_n65536", 1, 8, 65536, 3, 64, 64, 1024, 10, "bf16",
                      0.5, "uniform", "uniform", 2)
LONG = Workload("long_bf16_n1048576", 1, 8, 1048576, 3, 64, 64, 4096, 10, "bf16", 0.5,
                "uniform", "uniform", 3)
TRAIN = Workload("train_bf16_b4_n65536", 4, 8, 65536, 3, 64, 48, 1024, 10, "bf16", 0.5,
                 "uniform", "uniform", 4)

# The pages' own grid: 12 bits per coordinate, 36-bit codes (64-bit containers),
# at the efficiency scale.
PAGES12 = EFFICIENCY.replace(name="efficiency12_bf16_n65536", bits=12)

ALL = {w.name: w for w in (TINY, CLUSTERED, EFFICIENCY, LONG, TRAIN, PAGES12)}

# Locality side sweep: N=16384, C=1024, d_K in {1,2,3,8} at 21/21/10/8 bits.
SWEEP = [LONG.replace(name=f"sweep_dk{dk}_n16384", N=16384, C=1024, d_K=dk, bits=b)
         for dk, b in ((1, 21), (2, 21), (3, 10), (8, 8))]

# Finite-difference instance for the gradient check: the training workload's
# parameters at N=256, C=128.
FD = TRAIN.replace(name="fd_n256", B=1, H=2, N=256, C=128)


# Two-layer projection front end: token features of width D = H * d_V feed a
# per-head Linear(D -> F), ReLU, Linear(F -> d_K), tanh, for queries and keys.
@dataclasses.dataclass(frozen=True)
class Projection:
    name: str
    base: Workload        # B, H, N, d_K, bits (and the attention that follows)
    D: int
    F: int
    seed: int


PROJ = Projection("proj_train_b4_n65536_d512", TRAIN, 512, 64, 5)
PROJ_SMALL = Projection("proj_small", TRAIN.replace(B=1, H=4, N=1024, C=128), 128, 64, 6)


def generate_projection(pj: Projection) -> dict:
    """Draw x [B, N, D] ~ N(0, 1); per projection (query, key): W1 [H*F, D] ~
    N(0, 1/D), b1 [H*F] ~ N(0, 0.1^2), W2 [H, d_K, F] ~ N(0, 2/F), b2 [H, d_K] ~
    N(0, 0.1^2).  x and W1 are bf16 bit patterns (int16), stacked [2, ...] for
    (query, key); biases and W2 float32."""
    w = pj.base
    st = SplitMix64(pj.seed)
    x = st.normal_f64(w.B * w.N * pj.D).astype(np.float32).reshape(w.B, w.N, pj.D)
    HF = w.H * pj.F
    W1 = (st.normal_f64(2 * HF * pj.D) / np.sqrt(pj.D)).astype(np.float32).reshape(2, HF, pj.D)
    b1 = (0.1 * st.normal_f64(2 * HF)).astype(np.float32).reshape(2, HF)
    W2 = (st.normal_f64(2 * w.H * w.d_K * pj.F) * np.sqrt(2.0 / pj.F)).astype(np.float32)
    W2 = W2.reshape(2, w.H, w.d_K, pj.F)
    b2 = (0.1 * st.normal_f64(2 * w.H * w.d_K)).astype(np.float32).reshape(2, w.H, w.d_K)
    return {"x": f32_to_bf16_bits(x), "W1": f32_to_bf16_bits(W1), "b1": b1, "W2": W2, "b2": b2}


def _points(st: SplitMix64, w: Workload, count: int, centres: Optional[np.ndarray]) -> np.ndarray:
    if w.dist == "uniform":
        return st.uniform_pm1_f32(count * w.d_K).reshape(count, w.d_K)
    comp = np.minimum((st.uniform01_f64(count) * centres.shape[0]).astype(np.int64),
                      centres.shape[0] - 1)
    noise = st.normal_f64(count * w.d_K).reshape(count, w.d_K)
    x = (centres[comp] + 0.05 * noise).astype(np.float32)
    return np.clip(x, np.float32(-1.0), np.float32(1.0 - 2.0 ** -24))


def generate(w: Workload, with_dout: bool = False, dout_f32: bool = False) -> dict:
    """Draw q, k [B,H,N,d_K] f32; v [B,H,N,d_V]; gamma [H] f32; optional dO.

    v (and dO) are float32 for v_dtype 'f32', else bf16 bit patterns (int16);
    'v_f32' / 'dout_f32' always hold the unrounded float32 draws."""
    st = SplitMix64(w.seed)
    count = w.B * w.H * w.N
    centres = None
    if w.dist == "clusters":
        centres = -0.9 + 1.8 * st.uniform01_f64(64 * w.d_K).reshape(64, w.d_K)
    q = _points(st, w, count, centres).reshape(w.B, w.H, w.N, w.d_K)
    k = _points(st, w, count, centres).reshape(w.B, w.H, w.N, w.d_K)
    nv = count * w.d_V
    if w.v_dist == "uniform":
        v32 = st.uniform_pm1_f32(nv)
    else:
        v32 = st.normal_f64(nv).astype(np.float32)
    v32 = v32.reshape(w.B, w.H, w.N, w.d_V)
    if isinstance(w.gamma, tuple):
        lo, hi = w.gamma
        gamma = (lo + (hi - lo) * st.uniform01_f64(w.H)).astype(np.float32)
    else:
        gamma = np.full(w.H, w.gamma, dtype=np.float32)
    out = {"q": q, "k": k, "gamma": gamma, "v_f32": v32}
    out["v"] = v32 if w.v_dtype == "f32" else f32_to_bf16_bits(v32)
    if with_dout:
        d32 = st.normal_f64(nv).astype(np.float32).reshape(w.B, w.H, w.N, w.d_V)
        out["dout_f32"] = d32
        out["dout"] = d32 if (w.v_dtype == "f32" or dout_f32) else f32_to_bf16_bits(d32)
    return out


def values_f64(w: Workload, arr: np.ndarray) -> np.ndarray:
    """Widen a generated v / dO array (float32 or bf16 bits) to float64."""
    if arr.dtype == np.int16 or arr.dtype == np.uint16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return arr.astype(np.float64)
