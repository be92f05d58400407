"""The fast step without a workspace (sfi_fast_attn_noalloc).

Some callers cannot allocate device memory where the step runs -- a plug-in
interface that hands over only inputs and outputs, or a serving loop that
allocates nothing after start-up because cudaMalloc can synchronise the whole
device.  These tests run that entry point through the C ABI twice in a row and
check each result against the regular sfi_fast_attn (which takes a caller
workspace) within the parity tolerance of the fast step, and against the fp64
oracle's fast step.  The geometries include few (sequence, KV head) units with
a long managed state, where every unit is cut into many work pieces (the case
where the number of pieces per unit meets the merge's limit).  The file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import DeviceLayer, O_TOL, load_sfi, max_abs

pytestmark = pytest.mark.gpu


def _random_selection(rng, B, hkv, k, lens, n_sink, window):
    """A valid selection per (sequence, KV head): k_eff positions of the
    eligible range [n_sink, n - window), ascending (the fast step takes any
    such set; the selector is tested elsewhere)."""
    idx = np.zeros((B, hkv, k), np.int32)
    cnt = np.zeros((B, hkv), np.int32)
    for b in range(B):
        lo, hi = O.eligible_range(lens[b], n_sink, window)
        ke = min(k, hi - lo)
        for g in range(hkv):
            sel = np.sort(rng.choice(np.arange(lo, hi), size=ke, replace=False))
            idx[b, g, :ke] = sel
            cnt[b, g] = ke
    return idx, cnt


def _run_case(sfi, B, hq, hkv, d, dt, lens, k, window, seed, check_oracle):
    n_sink = 4
    wl = W.small(B, hq, hkv, d, dt, lens, seed=seed, n_sink=n_sink, window=window, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    qd, q64 = dl.queries(0)
    rng = np.random.default_rng(seed)
    idx_np, cnt_np = _random_selection(rng, B, hkv, k, lens, n_sink, window)
    idx = torch.from_numpy(idx_np).cuda()
    cnt = torch.from_numpy(cnt_np).cuda()
    prm = sfi.params(n_sink, window, k, 0.3)
    ws = sfi.alloc_workspace(lay)
    ref = torch.empty(B, hq, d, device="cuda")
    sfi.sfi_fast_attn(lay, prm, qd, dl.k, dl.v, idx, cnt, ref, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    ref = ref.cpu().numpy()
    exp = None
    if check_oracle:
        exp = np.stack([O.fast_step(q64[b], dl.K64[b], dl.V64[b], lens[b],
                                    [idx_np[b, g, :cnt_np[b, g]].astype(np.int64) for g in range(hkv)],
                                    n_sink, window) for b in range(B)])
        assert max_abs(ref, exp) <= O_TOL[dt]
    for call in range(2):
        got = torch.full((B, hq, d), float("nan"), device="cuda")
        sfi.sfi_fast_attn_noalloc(lay, prm, qd, dl.k, dl.v, idx, cnt, got)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        assert np.all(np.isfinite(got)), call
        err = max_abs(got, ref)
        assert err <= O_TOL[dt], (call, err)
        if exp is not None:
            err = max_abs(got, exp)
            assert err <= O_TOL[dt], (call, err)


def test_noalloc_fast_step_matches_workspace_version():
    sfi = load_sfi()
    _run_case(sfi, 3, 32, 8, 128, "bf16", [5000, 1200, 3333], 300, 256, 41, check_oracle=False)
    _run_case(sfi, 3, 32, 8, 128, "f32", [5000, 1200, 3333], 300, 256, 42, check_oracle=False)


# Few units and a long managed state: 1 or 2 units of n_sink + k + window =
# 4356 rows, cut into many work pieces each.
@pytest.mark.parametrize("hkv", [1, 2])
@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64)])
def test_noalloc_few_units_long_state_vs_oracle(hkv, dt, d):
    sfi = load_sfi()
    _run_case(sfi, 1, 4 * hkv, hkv, d, dt, [8192], 4096, 256, 50 + hkv, check_oracle=True)


def test_noalloc_rejects_oversized_geometry():
    sfi = load_sfi()
    L = sfi.sfi_layout(512, 64, 8, 128, sfi.SFI_BF16, 1000, 0x10000, 0x10000, 0x10000)
    p = sfi.params(4, 16, 8, 0.3)
    r = sfi.lib.sfi_fast_attn_noalloc(ctypes.byref(L), ctypes.byref(p), 0x10000, 0x10000, 0x10000,
                                      0x10000, 0x10000, 0x10000, None)
    assert r == sfi.SFI_ERR_CAPACITY
    assert "scratch" in sfi.lib.sfi_last_error().decode()
