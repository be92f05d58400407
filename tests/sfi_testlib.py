"""Shared helpers of the parity tests: device packing of seeded workloads, the
library calls through the binding, and the comparison rules.

Inputs come from ``sfi_workloads`` (the same stored bytes go to the GPU and,
as exact fp64 values, to the oracle); expected values come from ``oracle/``.
"""
from __future__ import annotations

import os
import sys
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import sfi_workloads as W
import oracle.sfi_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances stated for the path: attention outputs 1e-2 max-abs for bf16 KV and
# 2e-5 for fp32 KV; f and s 1e-5 absolute; selected sets identical except at
# positions whose score is within 1e-6 (relative) of the k-th value.  Key norms
# have no stated bound: 1e-5 relative follows from fp32 accumulation of at
# most 128 squares.
O_TOL = {"f32": 2e-5, "bf16": 1e-2}
F_TOL = 1e-5
S_TOL = 1e-5
KNORM_RTOL = 1e-5
TIE_RTOL = 1e-6


def load_sfi():
    """Import the binding, building the library first if it is missing."""
    lib = os.path.join(ROOT, "slow_sparse_kv_gb300", "_lib", "libsfi.so")
    if not os.path.exists(lib):
        sys.path.insert(0, ROOT)
        import __graft_entry__
        __graft_entry__.build()
    import slow_sparse_kv_gb300 as sfi
    return sfi


def storage_to_torch(arr: np.ndarray, dtype: str) -> torch.Tensor:
    arr = np.ascontiguousarray(arr)
    if dtype == "f32":
        return torch.from_numpy(arr.astype(np.float32, copy=False))
    return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)


def torch_dtype(dtype: str) -> torch.dtype:
    return torch.float32 if dtype == "f32" else torch.bfloat16


@dataclass
class DeviceLayer:
    """One layer's KV cache for every sequence of a workload, on the device,
    plus the exact fp64 values of the same stored elements for the oracle."""
    wl: W.Workload
    layer: int
    k: torch.Tensor
    v: torch.Tensor
    offsets: List[int]
    K64: List[np.ndarray]
    V64: List[np.ndarray]

    @staticmethod
    def build(wl: W.Workload, layer: int = 0, kv_override=None) -> "DeviceLayer":
        sh = wl.shape
        ks, vs, offs, K64, V64 = [], [], [], [], []
        off = 0
        for b in range(sh.batch):
            if kv_override is not None:
                kst, vst = kv_override(b)
            else:
                kst = wl.kv_storage("k", layer, b)
                vst = wl.kv_storage("v", layer, b)
            ks.append(storage_to_torch(kst, sh.dtype).reshape(-1))
            vs.append(storage_to_torch(vst, sh.dtype).reshape(-1))
            K64.append(W.storage_to_f64(kst, sh.dtype))
            V64.append(W.storage_to_f64(vst, sh.dtype))
            offs.append(off)
            off += kst.size
        return DeviceLayer(wl, layer, torch.cat(ks).cuda(), torch.cat(vs).cuda(), offs, K64, V64)

    def layout(self, sfi, lens, max_len: Optional[int] = None):
        sh = self.wl.shape
        ml = max_len if max_len is not None else max(self.wl.cap)
        return sfi.Layout(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, torch_dtype(sh.dtype),
                          self.offsets, self.wl.cap, lens, ml)

    def queries(self, step: int, row: int = 0):
        """(device q [B, H_q, d], list of fp64 [H_q, d] per sequence)."""
        sh = self.wl.shape
        sts = [self.wl.q_storage(self.layer, step, b, row) for b in range(sh.batch)]
        qd = torch.stack([storage_to_torch(s, sh.dtype) for s in sts]).cuda()
        return qd, [W.storage_to_f64(s, sh.dtype) for s in sts]


def check_selection(gpu_idx: np.ndarray, s_ref: np.ndarray, lo: int, hi: int, k: int,
                    rtol: float = TIE_RTOL, atol: float = 0.0) -> None:
    """The GPU set must have size min(k, |E|), be ascending, lie in E, and agree
    with the oracle's top-k on every position whose reference score is not
    within the tie band around the oracle's k-th value."""
    ke = max(0, min(k, hi - lo))
    assert len(gpu_idx) == ke, (len(gpu_idx), ke)
    if ke == 0:
        return
    assert np.all(np.diff(gpu_idx) > 0), "selection not strictly ascending"
    assert gpu_idx.min() >= lo and gpu_idx.max() < hi, "selection outside E"
    ref = O.top_k(s_ref, lo, hi, k)
    if ke == hi - lo:
        assert np.array_equal(gpu_idx, ref)
        return
    sc = s_ref[lo:hi]
    tau = np.sort(sc)[::-1][ke - 1]
    band = rtol * abs(tau) + atol
    amb = np.abs(s_ref - tau) <= band
    g = set(int(x) for x in gpu_idx)
    r = set(int(x) for x in ref)
    bad = [i for i in g.symmetric_difference(r) if not amb[i]]
    assert not bad, f"{len(bad)} non-ambiguous positions differ, e.g. {bad[:5]} (tau={tau})"


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0
