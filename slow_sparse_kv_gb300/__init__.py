"""Python binding of libsfi, the GB300 decode-attention hot path of Slow-Fast
Inference (SFI) with Vegas-style aggregated selection.

This module only marshals arguments: every step of the path runs in the CUDA
kernels of ``_lib/libsfi.so`` (built in-tree from ``csrc/`` by
``__graft_entry__.build()``).  Importing it without the built library raises
ImportError; there is no CPU fallback.  Functions carry the C names declared
in ``include/sfi.h`` and take torch tensors (device memory) or None for the
nullable pointers; ``stream`` is a torch.cuda.Stream, a raw cudaStream_t
handle, or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_size_t, c_uint32, c_void_p
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsfi.so")

SFI_OK, SFI_ERR_INVALID_ARG, SFI_ERR_UNSUPPORTED, SFI_ERR_CAPACITY, SFI_ERR_WORKSPACE, SFI_ERR_CUDA = range(6)
SFI_F32, SFI_BF16 = 0, 1
SFI_SELECT_FUSED, SFI_SELECT_LOGIT_SUM_SEQ, SFI_SELECT_LOGIT_SUM_HEAD = 0, 1, 2
SFI_DEV_LEN_OVER_CAP, SFI_DEV_BAD_INDEX, SFI_DEV_WAIT_TIMEOUT, SFI_DEV_ITEMS_OVERFLOW = 1, 2, 4, 8
SFI_DEV_REFINE = 16


class sfi_layout(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("dtype", c_int32), ("max_len", c_int32),
                ("kv_offset", c_void_p), ("kv_cap", c_void_p), ("len", c_void_p)]


class sfi_params(ctypes.Structure):
    _fields_ = [("n_sink", c_int32), ("window", c_int32), ("k", c_int32),
                ("lam", c_float), ("mode", c_int32)]


class sfi_refine(ctypes.Structure):
    _fields_ = [("nms_radius", c_int32), ("nms_sigma", c_float), ("excl_beta", c_float)]


class sfi_ctx_desc(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("dtype", c_int32), ("max_len", c_int32),
                ("n_layers", c_int32), ("params", sfi_params), ("budget", c_int32),
                ("async_select", c_int32), ("refine", sfi_refine)]


_L = POINTER(sfi_layout)
_P = POINTER(sfi_params)
# name -> (restype, argtypes); every function declared in include/sfi.h
EXPORTS = {
    "sfi_last_error": (c_char_p, []),
    "sfi_read_status": (c_int32, [c_void_p, POINTER(c_uint32), c_void_p]),
    "sfi_device_sm_count": (c_int32, []),
    "sfi_set_wait_limit": (c_int32, [ctypes.c_int64]),
    "sfi_slow_attn_workspace_size": (c_size_t, [_L]),
    "sfi_slow_attn": (c_int32, [_L, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_size_t, c_void_p]),
    "sfi_select_workspace_size": (c_size_t, [_L, _P]),
    "sfi_select": (c_int32, [_L, _P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_size_t, c_void_p]),
    "sfi_select_refined_workspace_size": (c_size_t, [_L, _P, POINTER(sfi_refine)]),
    "sfi_select_refined": (c_int32, [_L, _P, POINTER(sfi_refine), c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "sfi_fast_attn_workspace_size": (c_size_t, [_L, _P]),
    "sfi_fast_attn": (c_int32, [_L, _P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_size_t, c_void_p]),
    "sfi_verify_attn_workspace_size": (c_size_t, [_L, c_int32]),
    "sfi_verify_attn": (c_int32, [_L, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "sfi_fast_attn_noalloc": (c_int32, [_L, _P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p]),
    "sfi_ctx_create": (c_int32, [POINTER(sfi_ctx_desc), POINTER(c_void_p)]),
    "sfi_ctx_destroy": (c_int32, [c_void_p]),
    "sfi_decode_step": (c_int32, [c_void_p, c_int32, c_void_p, _L, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "sfi_schedule": (c_int32, [c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "sfi_ctx_reset": (c_int32, [c_void_p]),
    "sfi_ctx_read_status": (c_int32, [c_void_p, POINTER(c_uint32), c_void_p]),
    "sfi_ctx_profile": (c_int32, [c_void_p, c_int32]),
    "sfi_ctx_profile_read": (c_int32, [c_void_p, POINTER(ctypes.c_double), POINTER(ctypes.c_int64),
                                       POINTER(ctypes.c_double), POINTER(ctypes.c_int64)]),
    "sfi_ctx_slow_mask": (c_int32, [c_void_p, c_void_p]),
    "sfi_ctx_selection": (c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libsfi is not built ({LIB_PATH} missing): run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` first.  There is no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class SfiError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib.sfi_last_error().decode(errors="replace")
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != SFI_OK:
        raise SfiError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libsfi takes device tensors")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return SFI_F32
    if dt == torch.bfloat16:
        return SFI_BF16
    raise ValueError(f"unsupported dtype {dt}")


class Layout:
    """Batch/cache geometry of one layer: owns the device arrays the C layout points to.

    ``kv_offset[b]`` (elements), ``kv_cap[b]`` and ``len[b]`` describe where
    sequence b's [H_kv][cap][d] block lives and how long it is."""

    def __init__(self, n_q_heads: int, n_kv_heads: int, head_dim: int, dtype: torch.dtype,
                 kv_offset: Sequence[int], kv_cap: Sequence[int], lens: Sequence[int],
                 max_len: int, device="cuda"):
        self.B = len(kv_cap)
        self.n_q_heads, self.n_kv_heads, self.head_dim = n_q_heads, n_kv_heads, head_dim
        self.dtype = dtype
        self.max_len = int(max_len)
        self.kv_offset = torch.tensor(list(kv_offset), dtype=torch.int64, device=device)
        self.kv_cap = torch.tensor(list(kv_cap), dtype=torch.int32, device=device)
        self.len = torch.tensor(list(lens), dtype=torch.int32, device=device)
        self._c = None

    def set_lens(self, lens: Sequence[int]) -> None:
        self.len.copy_(torch.tensor(list(lens), dtype=torch.int32))

    @property
    def c(self) -> sfi_layout:
        return sfi_layout(self.B, self.n_q_heads, self.n_kv_heads, self.head_dim,
                          dtype_code(self.dtype), self.max_len, self.kv_offset.data_ptr(),
                          self.kv_cap.data_ptr(), self.len.data_ptr())


def params(n_sink: int, window: int, k: int, lam: float, mode: int = SFI_SELECT_FUSED) -> sfi_params:
    return sfi_params(int(n_sink), int(window), int(k), float(lam), int(mode))


def workspace_size(layout: Layout) -> int:
    c = layout.c
    return int(lib.sfi_slow_attn_workspace_size(ctypes.byref(c)))


def alloc_workspace(layout: Layout) -> torch.Tensor:
    """A zero-filled device workspace for every call of this geometry."""
    n = workspace_size(layout)
    if n == 0:
        raise SfiError("sfi_slow_attn_workspace_size", SFI_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def sfi_slow_attn(layout: Layout, q, k, v, out, f_out=None, knorm_out=None, ws=None, stream=None):
    c = layout.c
    _check("sfi_slow_attn", lib.sfi_slow_attn(
        ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(f_out), _ptr(knorm_out),
        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def sfi_select(layout: Layout, prm: sfi_params, evidence, knorm, idx_out, count_out, s_out=None,
               ws=None, stream=None):
    c = layout.c
    _check("sfi_select", lib.sfi_select(
        ctypes.byref(c), ctypes.byref(prm), _ptr(evidence), _ptr(knorm), _ptr(idx_out),
        _ptr(count_out), _ptr(s_out), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def sfi_select_refined(layout: Layout, prm: sfi_params, ref: sfi_refine, f, knorm, idx_out,
                       count_out, s_out=None, ws=None, stream=None):
    c = layout.c
    _check("sfi_select_refined", lib.sfi_select_refined(
        ctypes.byref(c), ctypes.byref(prm), ctypes.byref(ref), _ptr(f), _ptr(knorm), _ptr(idx_out),
        _ptr(count_out), _ptr(s_out), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def select_refined_workspace_size(layout: Layout, prm: sfi_params, ref: sfi_refine) -> int:
    return int(lib.sfi_select_refined_workspace_size(ctypes.byref(layout.c), ctypes.byref(prm),
                                                     ctypes.byref(ref)))


def sfi_fast_attn(layout: Layout, prm: sfi_params, q, k, v, idx, count, out, ws=None, stream=None):
    c = layout.c
    _check("sfi_fast_attn", lib.sfi_fast_attn(
        ctypes.byref(c), ctypes.byref(prm), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(count),
        _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def sfi_schedule(is_boundary, have_sel, since, budget: int):
    """Host-only schedule step on numpy arrays (uint8, uint8, int32; updated in place).
    Returns the slow mask (uint8 [B])."""
    import numpy as np
    B = len(is_boundary)
    ib = np.ascontiguousarray(is_boundary, np.uint8)
    out = np.zeros(B, np.uint8)
    assert have_sel.dtype == np.uint8 and since.dtype == np.int32
    _check("sfi_schedule", lib.sfi_schedule(B, int(budget), ib.ctypes.data, have_sel.ctypes.data,
                                            since.ctypes.data, out.ctypes.data))
    return out


def verify_workspace(layout: Layout, n_rows: int) -> torch.Tensor:
    """A zero-filled workspace for sfi_verify_attn with n_rows chain rows."""
    c = layout.c
    n = int(lib.sfi_verify_attn_workspace_size(ctypes.byref(c), int(n_rows)))
    if n == 0:
        raise SfiError("sfi_verify_attn_workspace_size", SFI_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def sfi_verify_attn(layout: Layout, n_rows: int, collect_rows, q, k, v, out, logitsum_out=None,
                    ws=None, stream=None):
    rows = list(collect_rows or [])
    arr = (c_int32 * max(1, len(rows)))(*rows)
    c = layout.c
    _check("sfi_verify_attn", lib.sfi_verify_attn(
        ctypes.byref(c), int(n_rows), arr, len(rows), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
        _ptr(logitsum_out), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def sfi_fast_attn_noalloc(layout: Layout, prm: sfi_params, q, k, v, idx, count, out, stream=None):
    """The fast step without a workspace (scratch in a fixed array inside the
    library), for callers that may not allocate on the path that runs it."""
    c = layout.c
    _check("sfi_fast_attn_noalloc", lib.sfi_fast_attn_noalloc(
        ctypes.byref(c), ctypes.byref(prm), _ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(count),
        _ptr(out), _stream(stream)))


def sfi_read_status(ws: torch.Tensor, stream=None) -> int:
    st = c_uint32(0)
    _check("sfi_read_status", lib.sfi_read_status(_ptr(ws), ctypes.byref(st), _stream(stream)))
    return int(st.value)


class DecodeContext:
    """sfi_ctx wrapper: per-layer selections plus the slow/fast schedule.

    ``refine`` (an ``sfi_refine``) applies Soft-NMS / cross-head exclusivity
    at every refresh; None keeps the plain Top-K."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, dtype: torch.dtype,
                 max_len: int, n_layers: int, prm: sfi_params, budget: int,
                 async_select: bool = True, refine: Optional[sfi_refine] = None):
        desc = sfi_ctx_desc(batch, n_q_heads, n_kv_heads, head_dim, dtype_code(dtype), max_len,
                            n_layers, prm, budget, int(bool(async_select)),
                            refine if refine is not None else sfi_refine(0, 0.0, 0.0))
        h = c_void_p()
        _check("sfi_ctx_create", lib.sfi_ctx_create(ctypes.byref(desc), ctypes.byref(h)))
        self.h = h
        self.batch, self.n_kv_heads, self.k = batch, n_kv_heads, prm.k

    def close(self) -> None:
        if self.h:
            lib.sfi_ctx_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def step(self, layer: int, is_boundary, layout: Layout, q, k, v, out, stream=None) -> None:
        """sfi_decode_step; is_boundary is a host uint8 sequence (read at layer 0)."""
        buf = None
        if is_boundary is not None:
            buf = (ctypes.c_uint8 * self.batch)(*[int(x) for x in is_boundary])
        c = layout.c
        _check("sfi_decode_step", lib.sfi_decode_step(
            self.h, int(layer), buf, ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
            _stream(stream)))

    def reset(self) -> None:
        _check("sfi_ctx_reset", lib.sfi_ctx_reset(self.h))

    def profile(self, enable: bool) -> None:
        _check("sfi_ctx_profile", lib.sfi_ctx_profile(self.h, int(bool(enable))))

    def profile_read(self):
        """(attention ms, attention launches, evidence+selector ms, their launches)."""
        am, sm = ctypes.c_double(), ctypes.c_double()
        al, sl = ctypes.c_int64(), ctypes.c_int64()
        _check("sfi_ctx_profile_read", lib.sfi_ctx_profile_read(
            self.h, ctypes.byref(am), ctypes.byref(al), ctypes.byref(sm), ctypes.byref(sl)))
        return am.value, al.value, sm.value, sl.value

    def read_status(self, stream=None) -> int:
        """OR of the context's device status words (cleared); waits for the stream."""
        v = c_uint32(0)
        _check("sfi_ctx_read_status", lib.sfi_ctx_read_status(self.h, ctypes.byref(v),
                                                              _stream(stream)))
        return int(v.value)

    def slow_mask(self):
        buf = (ctypes.c_uint8 * self.batch)()
        _check("sfi_ctx_slow_mask", lib.sfi_ctx_slow_mask(self.h, buf))
        return [int(x) for x in buf]

    def selection(self, layer: int, stream=None):
        """Copies of the layer's selection: (idx [B, H_kv, k], count [B, H_kv]) int32."""
        idx = torch.empty(self.batch, self.n_kv_heads, self.k, dtype=torch.int32, device="cuda")
        cnt = torch.empty(self.batch, self.n_kv_heads, dtype=torch.int32, device="cuda")
        _check("sfi_ctx_selection", lib.sfi_ctx_selection(self.h, int(layer), _ptr(idx), _ptr(cnt),
                                                          _stream(stream)))
        return idx, cnt
