"""Overlapped selection: a decode context whose selectors run on their own
stream beside the next layer's attention must give bit-identical outputs and
selections to one that runs them in line (same kernels, same inputs), over a
3-layer batch-8 decode at context 16384 with refreshes, budget expiries and
fast steps mixed in one launch."""
import pytest
import torch

import sfi_workloads as W
from tests.sfi_testlib import load_sfi

pytestmark = pytest.mark.gpu


def _run(sfi, R, wl, async_select):
    sh = wl.shape
    ctx = sfi.DecodeContext(sh.batch, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, torch.bfloat16,
                            R.max_len, wl.n_layers, sfi.params(wl.n_sink, wl.window, wl.k, wl.lam),
                            wl.budget, async_select=async_select)
    outs, sels, masks = [], [], []
    for t in range(wl.n_steps):
        for l in range(wl.n_layers):
            assert sfi.lib.sfi_decode_step(ctx.h, l, R.bnd[t], R.layouts[t], R.Q[l][t].data_ptr(),
                                           R.kp[l], R.vp[l], R.op[l], R.stream.cuda_stream) == 0
            outs.append(R.out[l].clone())
        masks.append(ctx.slow_mask())
        # every layer's selection after the token (ordered behind the selectors)
        sels.append([ctx.selection(l) for l in range(wl.n_layers)])
    assert ctx.read_status() == 0
    torch.cuda.synchronize()
    ctx.close()
    return outs, sels, masks


def test_async_select_bit_identical():
    assert torch.cuda.is_available()
    sfi = load_sfi()
    import bench
    wl = W.cfg2(n_layers=3, n_steps=24)
    wl.n0 = [16384] * 8
    wl.cap = [16384 + 256] * 8
    wl.k = 1024
    R = bench.Cfg2Runner(wl, 0)
    o_sync, s_sync, m_sync = _run(sfi, R, wl, False)
    o_async, s_async, m_async = _run(sfi, R, wl, True)
    assert m_sync == m_async
    assert any(any(m) and not all(m) for m in m_sync)  # some steps mix slow and fast
    for i, (x, y) in enumerate(zip(o_sync, o_async)):
        assert torch.equal(x, y), i
    for t in range(wl.n_steps):
        for l in range(wl.n_layers):
            (i0, c0), (i1, c1) = s_sync[t][l], s_async[t][l]
            assert torch.equal(c0, c1), (t, l)
            for b in range(wl.shape.batch):
                for g in range(wl.shape.n_kv_heads):
                    n = int(c0[b, g])
                    assert torch.equal(i0[b, g, :n], i1[b, g, :n]), (t, l, b, g)
