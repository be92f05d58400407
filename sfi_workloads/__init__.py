"""Seeded synthetic inputs for the SFI decode-attention hot path.

This module is the only code shared by the fp64 oracle (``oracle/``) and the
CUDA path (``slow_sparse_kv_gb300``).  It holds input generation only: shapes,
seeds, the counter-based normal generator, heavy-hitter planting and the
synthetic boundary traces.  It contains none of the method's arithmetic
(attention, evidence, prior, fusion, top-k, scheduling).

Counter-based normal generator (defined once, implemented here in numpy and in
``gen.cu`` for device-side fills of the very large workloads):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014; the constants
  are those of Vigna's public-domain ``splitmix64.c``).
* A stream key is ``key = mix64(seed + PHI)`` folded with each integer label
  ``key = mix64(key ^ (label + PHI))``; ``PHI = 0x9E3779B97F4A7C15``.
* Word ``c`` of a stream is ``w(c) = mix64(key + (c + 1) * PHI)`` (mod 2^64).
* Element ``e`` uses the pair ``p = e >> 1``: ``u1 = ((w(2p) >> 11) + 0.5) / 2^53``,
  ``u2 = (w(2p+1) >> 11) / 2^53``, ``rad = sqrt(-2 ln u1)``, and the
  Box-Muller transform gives ``rad*cos(2 pi u2)`` for even ``e`` and
  ``rad*sin(2 pi u2)`` for odd ``e``, in fp64.
* Stored values are rounded fp64 -> fp32 (round to nearest even) and, for bf16
  storage, fp32 -> bf16 (round to nearest even), the conversion torch uses too.

Workload recipe (the pages give no workload; these follow the synthetic
heavy-hitter recipe: K, V ~ N(0,1); 1% of positions get K += 3u for a fixed
random unit vector u; Q ~ N(0,1) + 2u):

* heavy positions: ``round(0.01 * cap)`` positions per (layer, sequence), drawn
  without replacement over the sequence's capacity; every KV head gets
  ``+3u`` at those positions;
* ``u``: one unit vector per layer, from the normal stream, normalised in fp64;
* K[l][b][g][i][j] = z + 3 u_j (heavy i) or z; V = z; Q[l][t][b][h][j] = z + 2 u_j;
  each tensor from its own stream, element index in row-major order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

PHI = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
MASTER_SEED = 20261202

# integer labels of the tensor streams
T_K, T_V, T_Q, T_U, T_HEAVY, T_TRACE, T_LENS, T_SLOWSET, T_IDX = 1, 2, 3, 4, 5, 6, 7, 8, 9


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def stream_key(seed: int, *labels: int) -> int:
    """Key of the stream named by ``labels`` under ``seed``."""
    k = mix64_int(seed + PHI)
    for lab in labels:
        k = mix64_int(k ^ ((int(lab) + PHI) & M64))
    return k


def _mix64_vec(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def normal_f64(key: int, start: int, count: int) -> np.ndarray:
    """fp64 standard normals for elements ``[start, start+count)`` of stream ``key``."""
    if count <= 0:
        return np.zeros(0, np.float64)
    e = np.arange(start, start + count, dtype=np.uint64)
    p = e >> np.uint64(1)
    with np.errstate(over="ignore"):
        c1 = (np.uint64(2) * p + np.uint64(1)) * np.uint64(PHI) + np.uint64(key)
        c2 = (np.uint64(2) * p + np.uint64(2)) * np.uint64(PHI) + np.uint64(key)
        w1 = _mix64_vec(c1)
        w2 = _mix64_vec(c2)
    u1 = ((w1 >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u2 = (w2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    rad = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    odd = (e & np.uint64(1)).astype(bool)
    return np.where(odd, rad * np.sin(th), rad * np.cos(th))


# ---------------------------------------------------------------- storage dtypes

def f64_to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, np.float64).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16))
    return u.view(np.float32).astype(np.float64)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to the storage dtype: float32 array, or uint16 bf16 bits."""
    x32 = f64_to_f32(x64)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 value of stored elements (bf16 and fp32 both embed exactly)."""
    if dtype == "f32":
        return np.asarray(a, np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    raise ValueError(dtype)


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Shape:
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str  # "f32" or "bf16"

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2


@dataclass
class Workload:
    """One synthetic workload.

    ``n0[b]`` is sequence b's cache length (including the current token) at the
    first decode step; step t runs at length ``n0[b] + t``.  ``cap[b]`` is the
    per-sequence capacity (positions) of the KV cache.
    """
    name: str
    cfg_id: int
    shape: Shape
    n_layers: int
    n0: List[int]
    cap: List[int]
    n_steps: int
    n_sink: int
    window: int
    k: int
    lam: float
    budget: int  # fast steps allowed between refreshes (0 = unlimited)
    seed: int = MASTER_SEED
    boundary_rate: float = 0.0  # per-step boundary probability (0: use fixed trace)
    fixed_slow_steps: Tuple[int, ...] = ()
    gamma: int = 0  # Vegas draft length (0: SFI workload)
    heavy_frac: float = 0.01
    notes: str = ""

    # ---------------------------------------------------------- keys
    def key(self, *labels: int) -> int:
        return stream_key(self.seed, self.cfg_id, *labels)

    def u_vec(self, layer: int) -> np.ndarray:
        """The layer's heavy-hitter direction u (fp64 unit vector)."""
        z = normal_f64(self.key(T_U, layer), 0, self.shape.head_dim)
        return z / np.sqrt(np.sum(z * z))

    def heavy_positions(self, layer: int, b: int) -> np.ndarray:
        cap = self.cap[b]
        m = int(round(self.heavy_frac * cap))
        rng = np.random.Generator(np.random.PCG64(self.key(T_HEAVY, layer, b)))
        return np.sort(rng.choice(cap, size=m, replace=False)).astype(np.int64)

    def heavy_mask(self, layer: int, b: int) -> np.ndarray:
        m = np.zeros(self.cap[b], dtype=bool)
        m[self.heavy_positions(layer, b)] = True
        return m

    # ---------------------------------------------------------- K / V / Q
    def kv_f64(self, which: str, layer: int, b: int, g: int, pos0: int = 0,
               npos: Optional[int] = None) -> np.ndarray:
        """fp64 pre-rounding values of K or V rows [pos0, pos0+npos) of head g: [npos, d]."""
        d = self.shape.head_dim
        cap = self.cap[b]
        if npos is None:
            npos = cap - pos0
        lab = T_K if which == "k" else T_V
        z = normal_f64(self.key(lab, layer, b), (g * cap + pos0) * d, npos * d).reshape(npos, d)
        if which == "k":
            hm = self.heavy_mask(layer, b)[pos0:pos0 + npos]
            z = z + np.where(hm[:, None], 3.0 * self.u_vec(layer)[None, :], 0.0)
        return z

    def kv_storage(self, which: str, layer: int, b: int, g: Optional[int] = None,
                   pos0: int = 0, npos: Optional[int] = None) -> np.ndarray:
        """Stored K or V of one sequence: [H_kv, npos, d] (or [npos, d] for one head)."""
        heads = range(self.shape.n_kv_heads) if g is None else [g]
        out = [to_storage(self.kv_f64(which, layer, b, hh, pos0, npos), self.shape.dtype)
               for hh in heads]
        return out[0] if g is not None else np.stack(out)

    def q_f64(self, layer: int, step: int, b: int, row: int = 0) -> np.ndarray:
        """fp64 pre-rounding query of decode step ``step`` (verify row ``row``): [H_q, d]."""
        hq, d = self.shape.n_q_heads, self.shape.head_dim
        z = normal_f64(self.key(T_Q, layer, b, step, row), 0, hq * d).reshape(hq, d)
        return z + 2.0 * self.u_vec(layer)[None, :]

    def q_storage(self, layer: int, step: int, b: int, row: int = 0) -> np.ndarray:
        return to_storage(self.q_f64(layer, step, b, row), self.shape.dtype)

    # ---------------------------------------------------------- traces
    def boundary_trace(self) -> np.ndarray:
        """is_boundary[step][b] (uint8): synthetic sentence-boundary events."""
        B, T = self.shape.batch, self.n_steps
        tr = np.zeros((T, B), np.uint8)
        if self.boundary_rate > 0:
            for b in range(B):
                rng = np.random.Generator(np.random.PCG64(self.key(T_TRACE, b)))
                tr[:, b] = (rng.random(T) < self.boundary_rate).astype(np.uint8)
        for t in self.fixed_slow_steps:
            if t < T:
                tr[t, :] = 1
        return tr


def cfg0() -> Workload:
    """Single layer, batch 1, 8 query / 2 KV heads, d=64, fp32, context 2048:
    one slow step then 16 fast steps; 4 sinks, window 256, k=128, lambda 0.3."""
    return Workload(name="gqa8x2-d64-f32-ctx2k", cfg_id=0,
                    shape=Shape(1, 8, 2, 64, "f32"), n_layers=1,
                    n0=[2048], cap=[2048 + 16], n_steps=17, n_sink=4, window=256,
                    k=128, lam=0.3, budget=0, fixed_slow_steps=(0,))


def cfg1() -> Workload:
    """Llama-3-8B-shaped layer (32/8 heads, d=128), bf16, batch 1, context 32768:
    64 decode steps, slow every 24 tokens, k=2048, window 256, 4 sinks, lambda 0.3."""
    return Workload(name="llama3-8b-layer-bf16-ctx32k", cfg_id=1,
                    shape=Shape(1, 32, 8, 128, "bf16"), n_layers=1,
                    n0=[32768], cap=[32768 + 64], n_steps=64, n_sink=4, window=256,
                    k=2048, lam=0.3, budget=0, fixed_slow_steps=(0, 24, 48))


def cfg2(n_layers: int = 32, n_steps: int = 256) -> Workload:
    """Same layer shape, bf16, context 131072, batch 8, 32 layers, 256 decode
    steps; boundaries geometric with mean 20 tokens, refresh budget 32, k=4096."""
    return Workload(name="llama3-8b-32L-bf16-b8-ctx128k", cfg_id=2,
                    shape=Shape(8, 32, 8, 128, "bf16"), n_layers=n_layers,
                    n0=[131072] * 8, cap=[131072 + 256] * 8, n_steps=n_steps, n_sink=4,
                    window=256, k=4096, lam=0.3, budget=32, boundary_rate=1.0 / 20.0)


def cfg3() -> Workload:
    """Vegas-style selection: same layer shape, bf16, prefix 65536, batch 4,
    draft length 4 (5 verify rows), Collect-2 rows {0, 4}, k=2048, 4 draft steps."""
    g = 4
    return Workload(name="vegas-llama3-8b-bf16-b4-ctx64k", cfg_id=3,
                    shape=Shape(4, 32, 8, 128, "bf16"), n_layers=1,
                    n0=[65536] * 4, cap=[65536 + 2 * g + 1] * 4, n_steps=1 + g,
                    n_sink=0, window=0, k=2048, lam=0.0, budget=0, gamma=g)


def cfg4_lengths(seed: int = MASTER_SEED, n_seq: int = 32) -> List[int]:
    rng = np.random.Generator(np.random.PCG64(stream_key(seed, 4, T_LENS)))
    x = rng.uniform(math.log(4096), math.log(262144), size=n_seq)
    return [int(round(math.exp(v))) for v in x]


def cfg4(k: int = 4096, window: int = 256) -> Workload:
    """Ragged serving batch: 32 sequences, contexts log-uniform in [4096, 262144],
    bf16 Llama-3-8B attention shape, 25% of sequences at a boundary."""
    lens = cfg4_lengths()
    return Workload(name=f"ragged32-llama3-8b-bf16-k{k}-w{window}", cfg_id=4,
                    shape=Shape(32, 32, 8, 128, "bf16"), n_layers=1,
                    n0=[n - 1 for n in lens], cap=lens, n_steps=2, n_sink=4,
                    window=window, k=k, lam=0.3, budget=0)


def cfg4_slow_set(seed: int = MASTER_SEED, n_seq: int = 32, n_slow: int = 8) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(stream_key(seed, 4, T_SLOWSET)))
    return np.sort(rng.choice(n_seq, size=n_slow, replace=False))


def small(B: int, hq: int, hkv: int, d: int, dtype: str, lens: Sequence[int], seed: int,
          n_sink: int = 4, window: int = 16, k: int = 8, lam: float = 0.3,
          n_steps: int = 4, extra: int = 8) -> Workload:
    """Small randomised workload for parity tests (ragged lengths allowed)."""
    lens = list(int(x) for x in lens)
    return Workload(name=f"small-{B}x{hq}x{hkv}x{d}-{dtype}-s{seed}", cfg_id=100 + seed % 1000,
                    shape=Shape(B, hq, hkv, d, dtype), n_layers=1, n0=lens,
                    cap=[n + extra for n in lens], n_steps=n_steps, n_sink=n_sink,
                    window=window, k=k, lam=lam, budget=0, seed=seed,
                    fixed_slow_steps=(0,))


WORKLOADS = {"cfg0": cfg0, "cfg1": cfg1, "cfg2": cfg2, "cfg3": cfg3, "cfg4": cfg4}
