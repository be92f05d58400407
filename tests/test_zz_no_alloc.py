"""The fast step without a workspace (sfi_fast_attn_noalloc).

Some callers cannot allocate device memory where the step runs -- a plug-in
interface that hands over only inputs and outputs, or a serving loop that
allocates nothing after start-up because cudaMalloc can synchronise the whole
device.  This test runs that entry point through the C ABI twice in a row and
checks each result against the regular sfi_fast_attn (which takes a caller
workspace) within the parity tolerance of the fast step.  The file is named to
be collected last.
"""
import numpy as np
import pytest
import torch

import sfi_workloads as W
from tests.sfi_testlib import DeviceLayer, O_TOL, load_sfi, max_abs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_noalloc_fast_step_matches_workspace_version(dt):
    assert torch.cuda.is_available()
    sfi = load_sfi()
    B, hq, hkv, d, k = 3, 32, 8, 128, 300
    lens = [5000, 1200, 3333]
    wl = W.small(B, hq, hkv, d, dt, lens, seed=41, n_sink=4, window=256, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, _ = dl.queries(0)
    f = torch.empty(B, hkv, lay.max_len, device="cuda")
    kn = torch.empty_like(f)
    out = torch.empty(B, hq, d, device="cuda")
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, f, kn, ws)
    prm = sfi.params(4, 256, k, 0.3)
    idx = torch.empty(B, hkv, k, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, hkv, dtype=torch.int32, device="cuda")
    sfi.sfi_select(lay, prm, f, kn, idx, cnt, None, ws)
    ref = torch.empty(B, hq, d, device="cuda")
    sfi.sfi_fast_attn(lay, prm, qd, dl.k, dl.v, idx, cnt, ref, ws)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    for call in range(2):
        got = torch.full((B, hq, d), float("nan"), device="cuda")
        sfi.sfi_fast_attn_noalloc(lay, prm, qd, dl.k, dl.v, idx, cnt, got)
        torch.cuda.synchronize()
        err = max_abs(got.cpu().numpy(), ref)
        assert err <= O_TOL[dt], (call, err)


def test_noalloc_rejects_oversized_geometry():
    sfi = load_sfi()
    import ctypes
    L = sfi.sfi_layout(512, 64, 8, 128, sfi.SFI_BF16, 1000, 0x10000, 0x10000, 0x10000)
    p = sfi.params(4, 16, 8, 0.3)
    r = sfi.lib.sfi_fast_attn_noalloc(ctypes.byref(L), ctypes.byref(p), 0x10000, 0x10000, 0x10000,
                                      0x10000, 0x10000, 0x10000, None)
    assert r == sfi.SFI_ERR_CAPACITY
    assert "scratch" in sfi.lib.sfi_last_error().decode()
