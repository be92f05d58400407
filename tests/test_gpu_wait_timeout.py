"""Failure detection on the GPU without a fault: a pipeline or barrier wait that runs out.

Every consumer wait of the attention kernel for a stage of cache rows has a
limit (sfi_set_wait_limit; about 2 s by default).  Here the limit is set to a
single SM clock, so the first wait for rows that have not landed yet gives up
(a CTA's first stage is never in shared memory when its consumers first look):
the kernel must set SFI_DEV_WAIT_TIMEOUT, return (the stream completes), and
leave the context usable -- after the workspace is zero-filled again, the same
call with the default limit must reproduce the oracle's dense output and the
bytes of a run made before the timeout.  No wait is left unbounded and nothing
faults: the copies a CTA issued still land before it exits."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import DeviceLayer, O_TOL, load_sfi, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture()
def sfi():
    assert torch.cuda.is_available()
    s = load_sfi()
    yield s
    assert s.lib.sfi_set_wait_limit(0) == s.SFI_OK


def test_wait_runs_out_then_recovers(sfi):
    lens = [40000, 23456]
    wl = W.small(2, 32, 8, 128, "bf16", lens, seed=77, n_sink=4, window=256, k=512)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, q64 = dl.queries(0)
    before = torch.empty(2, 32, 128, device="cuda")
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, before, None, None, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0

    assert sfi.lib.sfi_set_wait_limit(1) == sfi.SFI_OK
    out = torch.zeros(2, 32, 128, device="cuda")
    for _ in range(2):  # a second aborted launch on the dirty workspace also returns
        sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, None, None, ws)
        torch.cuda.synchronize()
        st = sfi.sfi_read_status(ws)
        assert st & sfi.SFI_DEV_WAIT_TIMEOUT, st

    assert sfi.lib.sfi_set_wait_limit(0) == sfi.SFI_OK
    ws.zero_()
    after = torch.empty(2, 32, 128, device="cuda")
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, after, None, None, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    assert torch.equal(after, before)
    for b in range(2):
        exp = O.dense_attention(q64[b], dl.K64[b], dl.V64[b], lens[b])[0]
        assert max_abs(after[b].cpu().numpy(), exp) <= O_TOL["bf16"]


def test_selector_barrier_wait_runs_out_then_recovers(sfi):
    """The selector's chunk CTAs of a unit wait for one another at barriers
    with the same limit.  One sequence x 8 KV heads at 40000 positions splits
    every unit into 20 chunk CTAs; with a one-clock limit the waits give up:
    SFI_DEV_WAIT_TIMEOUT is set, every access stays in bounds (the counts the
    CTAs then read are inconsistent) and the launch returns.  After the
    workspace is zero-filled again, the default limit reproduces the bytes of
    a selection made before the timeout."""
    lens = [40000]
    wl = W.small(1, 32, 8, 128, "bf16", lens, seed=78, n_sink=4, window=256, k=512)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, _ = dl.queries(0)
    out = torch.empty(1, 32, 128, device="cuda")
    f = torch.empty(1, 8, lay.max_len, device="cuda")
    kn = torch.empty(1, 8, lay.max_len, device="cuda")
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, f, kn, ws)
    prm = sfi.params(4, 256, 512, wl.lam)
    idx0 = torch.full((1, 8, 512), -1, dtype=torch.int32, device="cuda")
    cnt0 = torch.full((1, 8), -1, dtype=torch.int32, device="cuda")
    sfi.sfi_select(lay, prm, f, kn, idx0, cnt0, None, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0

    assert sfi.lib.sfi_set_wait_limit(1) == sfi.SFI_OK
    idx = torch.full_like(idx0, -1)
    cnt = torch.full_like(cnt0, -1)
    for _ in range(2):  # a second launch on the dirty workspace also returns
        sfi.sfi_select(lay, prm, f, kn, idx, cnt, None, ws)
        torch.cuda.synchronize()
        st = sfi.sfi_read_status(ws)
        assert st & sfi.SFI_DEV_WAIT_TIMEOUT, st

    assert sfi.lib.sfi_set_wait_limit(0) == sfi.SFI_OK
    ws.zero_()
    idx.fill_(-1)
    cnt.fill_(-1)
    sfi.sfi_select(lay, prm, f, kn, idx, cnt, None, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    assert torch.equal(cnt, cnt0)
    assert torch.equal(idx, idx0)
