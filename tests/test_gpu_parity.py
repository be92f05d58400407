"""GPU parity of the slow step, the selector and the fast step against the
fp64 oracle, element by element, through the C ABI (binding)."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import (DeviceLayer, F_TOL, KNORM_RTOL, O_TOL, S_TOL, check_selection,
                               load_sfi, max_abs, torch_dtype)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sfi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return load_sfi()


# (B, H_q, H_kv, d, dtype, lens, n_sink, window, k, seed)
CASES = [
    (3, 8, 2, 64, "f32", [37, 600, 1500], 4, 16, 20, 1),
    (2, 32, 8, 128, "bf16", [700, 2500], 4, 64, 100, 2),
    (2, 4, 4, 128, "f32", [300, 1], 2, 8, 5, 3),          # G = 1; a length-1 sequence
    (2, 16, 2, 64, "bf16", [1000, 333], 0, 10, 50, 4),     # G = 8, no sinks
    (1, 4, 2, 128, "bf16", [3000], 4, 256, 6000, 5),       # k >= |E|: keep all of E
    (2, 8, 4, 64, "f32", [40, 10], 4, 16, 8, 6),           # E empty for the second sequence
    (4, 8, 4, 128, "f32", [129, 257, 513, 1025], 1, 1, 1, 7),  # k = 1, window 1
    (1, 16, 8, 64, "f32", [4099], 4, 100, 700, 8),         # ragged tail past several stages
]


def ids(c):
    return f"B{c[0]}-hq{c[1]}-hkv{c[2]}-d{c[3]}-{c[4]}-k{c[8]}"


def run_slow(sfi, dl, lens, step=0):
    wl = dl.wl
    sh = wl.shape
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, q64 = dl.queries(step)
    out = torch.empty(sh.batch, sh.n_q_heads, sh.head_dim, device="cuda")
    f = torch.full((sh.batch, sh.n_kv_heads, lay.max_len), -7.0, device="cuda")
    kn = torch.full_like(f, -7.0)
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, f, kn, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    return lay, ws, q64, out.cpu().numpy(), f.cpu().numpy(), kn.cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_slow_select_fast_parity(sfi, case):
    B, hq, hkv, d, dt, lens, ns, win, k, seed = case
    wl = W.small(B, hq, hkv, d, dt, lens, seed, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay, ws, q64, out, f, kn = run_slow(sfi, dl, lens)
    prm = sfi.params(ns, win, k, wl.lam)
    idx = torch.full((B, hkv, k), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, hkv), -1, dtype=torch.int32, device="cuda")
    s = torch.full((B, hkv, lay.max_len), -7.0, device="cuda")
    f_d = torch.from_numpy(f).cuda()
    kn_d = torch.from_numpy(kn).cuda()
    sfi.sfi_select(lay, prm, f_d, kn_d, idx, cnt, s, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    idx, cnt, s = idx.cpu().numpy(), cnt.cpu().numpy(), s.cpu().numpy()
    for b in range(B):
        n = lens[b]
        st = O.slow_step(q64[b], dl.K64[b], dl.V64[b], n, ns, win, k, wl.lam)
        assert max_abs(out[b], st["o"]) <= O_TOL[dt], max_abs(out[b], st["o"])
        assert max_abs(f[b, :, :n], st["f"]) <= F_TOL
        np.testing.assert_allclose(kn[b, :, :n], st["knorm"], rtol=KNORM_RTOL, atol=1e-6)
        assert np.all(f[b, :, n:] == -7.0), "wrote past n"
        assert max_abs(s[b, :, :n], st["s"]) <= S_TOL
        lo, hi = st["lo"], st["hi"]
        for g in range(hkv):
            got = idx[b, g, :cnt[b, g]]
            check_selection(got, st["s"][g], lo, hi, k)
            # exact integer work in the kernel's precision: the set is the top-k
            # of the GPU's own fp32 scores under the tie rule
            assert np.array_equal(got, O.top_k(s[b, g].astype(np.float64), lo, hi, k))
    # fast steps with the GPU's selection at the slow length and two tokens later
    for extra in (0, 2):
        lens2 = [min(n + extra, c) for n, c in zip(lens, wl.cap)]
        lay2 = dl.layout(sfi, lens2)
        qd, q64f = dl.queries(1 + extra)
        out2 = torch.empty(B, hq, d, device="cuda")
        sfi.sfi_fast_attn(lay2, prm, qd, dl.k, dl.v, torch.from_numpy(idx).cuda(),
                          torch.from_numpy(cnt).cuda(), out2, ws)
        torch.cuda.synchronize()
        assert sfi.sfi_read_status(ws) == 0
        out2 = out2.cpu().numpy()
        for b in range(B):
            sel = [idx[b, g, :cnt[b, g]].astype(np.int64) for g in range(hkv)]
            ref = O.fast_step(q64f[b], dl.K64[b], dl.V64[b], lens2[b], sel, ns, win)
            assert max_abs(out2[b], ref) <= O_TOL[dt], (extra, b, max_abs(out2[b], ref))


def test_fast_all_positions_equals_dense(sfi):
    """k >= |E| at the slow step's length: the fast output equals the dense one."""
    wl = W.small(2, 8, 2, 128, "bf16", [900, 2000], 11, n_sink=4, window=32, k=4096)
    dl = DeviceLayer.build(wl)
    lens = [900, 2000]
    lay, ws, q64, out, f, kn = run_slow(sfi, dl, lens, step=0)
    prm = sfi.params(4, 32, 4096, 0.3)
    idx = torch.empty(2, 2, 4096, dtype=torch.int32, device="cuda")
    cnt = torch.empty(2, 2, dtype=torch.int32, device="cuda")
    sfi.sfi_select(lay, prm, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(), idx, cnt, None, ws)
    qd, _ = dl.queries(0)
    out2 = torch.empty_like(torch.from_numpy(out)).cuda()
    sfi.sfi_fast_attn(lay, prm, qd, dl.k, dl.v, idx, cnt, out2, ws)
    torch.cuda.synchronize()
    # same rows, different split points and P rounding: equal within the bf16 parity bar
    assert float((out2.cpu() - torch.from_numpy(out)).abs().max()) <= O_TOL["bf16"]


def test_ties_go_to_lower_positions(sfi):
    """Identical keys: f, r and s are flat, so the selection is the lowest positions of E."""
    B, hq, hkv, d = 1, 8, 2, 64
    n = 700
    wl = W.small(B, hq, hkv, d, "f32", [n], 12, n_sink=4, window=50, k=33)
    row = np.linspace(-1, 1, d).astype(np.float32)

    def kv(b):
        cap = wl.cap[b]
        k = np.broadcast_to(row, (hkv, cap, d)).copy()
        v = W.to_storage(np.random.default_rng(3).standard_normal((hkv, cap, d)), "f32")
        return k, v

    dl = DeviceLayer.build(wl, kv_override=kv)
    lay, ws, q64, out, f, kn = run_slow(sfi, dl, [n])
    prm = sfi.params(4, 50, 33, 0.3)
    idx = torch.empty(B, hkv, 33, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, hkv, dtype=torch.int32, device="cuda")
    sfi.sfi_select(lay, prm, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(), idx, cnt, None, ws)
    torch.cuda.synchronize()
    for g in range(hkv):
        assert list(idx[0, g].cpu().numpy()) == list(range(4, 37))


def test_bad_index_is_flagged_not_faulted(sfi):
    """A selected position outside [0, n) is skipped safely and reported."""
    wl = W.small(1, 8, 2, 64, "f32", [400], 13, n_sink=4, window=16, k=4)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, [400])
    ws = sfi.alloc_workspace(lay)
    qd, _ = dl.queries(0)
    idx = torch.tensor([[[10, 20, 30, 10 ** 6], [5, 6, 7, 8]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[4, 4]], dtype=torch.int32, device="cuda")
    out = torch.empty(1, 8, 64, device="cuda")
    sfi.sfi_fast_attn(lay, sfi.params(4, 16, 4, 0.3), qd, dl.k, dl.v, idx, cnt, out, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) & sfi.SFI_DEV_BAD_INDEX
    assert sfi.sfi_read_status(ws) == 0  # reading clears it


def test_length_over_capacity_is_flagged(sfi):
    wl = W.small(2, 8, 2, 64, "f32", [100, 50], 14, n_sink=4, window=16, k=4)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, [100, wl.cap[1] + 5], max_len=max(wl.cap) + 10)
    ws = sfi.alloc_workspace(lay)
    qd, _ = dl.queries(0)
    out = torch.zeros(2, 8, 64, device="cuda")
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, None, None, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) & sfi.SFI_DEV_LEN_OVER_CAP


@pytest.mark.parametrize("async_select", [False, True])
def test_decode_loop_cfg0(sfi, async_select):
    """The decode driver over the 17-step fp32 workload (1 slow + 16 fast)."""
    wl = W.cfg0()
    sh = wl.shape
    dl = DeviceLayer.build(wl)
    trace = wl.boundary_trace()
    slow_ref = O.schedule(trace, wl.budget)
    ctx = sfi.DecodeContext(sh.batch, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, torch.float32,
                            max(wl.cap), 1, sfi.params(wl.n_sink, wl.window, wl.k, wl.lam), wl.budget,
                            async_select=async_select)
    lay = dl.layout(sfi, wl.n0)
    qs64 = []
    outs = []
    for t in range(wl.n_steps):
        lay.set_lens([n + t for n in wl.n0])
        qd, q64 = dl.queries(t)
        qs64.append(q64[0])
        out = torch.empty(sh.batch, sh.n_q_heads, sh.head_dim, device="cuda")
        ctx.step(0, trace[t], lay, qd, dl.k, dl.v, out)
        assert ctx.slow_mask() == [int(x) for x in slow_ref[t]]
        outs.append(out.cpu().numpy()[0])
    torch.cuda.synchronize()
    ref = O.decode_sequence(qs64, dl.K64[0], dl.V64[0], wl.n0[0], slow_ref[:, 0], wl.n_sink,
                            wl.window, wl.k, wl.lam)
    idx_g, cnt_g = ctx.selection(0)
    idx_g, cnt_g = idx_g.cpu().numpy(), cnt_g.cpu().numpy()
    st = ref[0]
    for g in range(sh.n_kv_heads):
        check_selection(idx_g[0, g, :cnt_g[0, g]], st["s"][g], st["lo"], st["hi"], wl.k)
    sel = [idx_g[0, g, :cnt_g[0, g]].astype(np.int64) for g in range(sh.n_kv_heads)]
    for t in range(wl.n_steps):
        if ref[t]["kind"] == "slow":
            exp = ref[t]["o"]
        else:
            exp = O.fast_step(qs64[t], dl.K64[0], dl.V64[0], wl.n0[0] + t, sel, wl.n_sink, wl.window)
        assert max_abs(outs[t], exp) <= O_TOL["f32"], (t, max_abs(outs[t], exp))
    assert ctx.read_status() == 0
    ctx.close()


@pytest.fixture(scope="module")
def cfg1_layer():
    """The 32K-context Llama-3-8B layer of the cfg1 workload on the device (and
    its exact fp64 values for the oracle)."""
    return DeviceLayer.build(W.cfg1())


def test_cfg1_slow_select_fast(sfi, cfg1_layer):
    """Llama-3-8B layer, bf16, 32K context: slow step, selection and fast steps."""
    dl = cfg1_layer
    wl = dl.wl
    sh = wl.shape
    n = wl.n0[0]
    lay, ws, q64, out, f, kn = run_slow(sfi, dl, [n])
    st = O.slow_step(q64[0], dl.K64[0], dl.V64[0], n, wl.n_sink, wl.window, wl.k, wl.lam)
    assert max_abs(out[0], st["o"]) <= O_TOL["bf16"]
    assert max_abs(f[0, :, :n], st["f"]) <= F_TOL
    np.testing.assert_allclose(kn[0, :, :n], st["knorm"], rtol=KNORM_RTOL)
    prm = sfi.params(wl.n_sink, wl.window, wl.k, wl.lam)
    idx = torch.empty(1, sh.n_kv_heads, wl.k, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, sh.n_kv_heads, dtype=torch.int32, device="cuda")
    s = torch.empty(1, sh.n_kv_heads, lay.max_len, device="cuda")
    sfi.sfi_select(lay, prm, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(), idx, cnt, s, ws)
    torch.cuda.synchronize()
    s_np = s.cpu().numpy()
    assert max_abs(s_np[0, :, :n], st["s"]) <= S_TOL
    idx_np, cnt_np = idx.cpu().numpy(), cnt.cpu().numpy()
    for g in range(sh.n_kv_heads):
        check_selection(idx_np[0, g, :cnt_np[0, g]], st["s"][g], st["lo"], st["hi"], wl.k)
    sel = [idx_np[0, g, :cnt_np[0, g]].astype(np.int64) for g in range(sh.n_kv_heads)]
    for t in (1, 23):
        lay.set_lens([n + t])
        qd, qf = dl.queries(t)
        o2 = torch.empty(1, sh.n_q_heads, sh.head_dim, device="cuda")
        sfi.sfi_fast_attn(lay, prm, qd, dl.k, dl.v, idx, cnt, o2, ws)
        torch.cuda.synchronize()
        ref = O.fast_step(qf[0], dl.K64[0], dl.V64[0], n + t, sel, wl.n_sink, wl.window)
        assert max_abs(o2.cpu().numpy()[0], ref) <= O_TOL["bf16"]
    assert sfi.sfi_read_status(ws) == 0


def test_cfg1_decode_loop_64_steps(sfi, cfg1_layer):
    """The whole 64-step cfg1 loop through the decode driver: refreshes at
    steps 0, 24 and 48 (fixed boundary trace), fast steps between them.  Each
    refreshed selection must match the oracle's slow step (tie rule), each
    slow output its dense attention, and each fast output the oracle's fast
    step over the set the GPU held at that step."""
    dl = cfg1_layer
    wl = dl.wl
    sh = wl.shape
    trace = wl.boundary_trace()
    slow_ref = O.schedule(trace, wl.budget)
    assert [t for t in range(wl.n_steps) if slow_ref[t, 0]] == [0, 24, 48]
    ctx = sfi.DecodeContext(sh.batch, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, torch.bfloat16,
                            max(wl.cap), 1, sfi.params(wl.n_sink, wl.window, wl.k, wl.lam),
                            wl.budget, async_select=True)
    lay = dl.layout(sfi, wl.n0)
    outs, q64s, sels = [], [], {}
    for t in range(wl.n_steps):
        lay.set_lens([n + t for n in wl.n0])
        qd, q64 = dl.queries(t)
        q64s.append(q64[0])
        out = torch.empty(sh.batch, sh.n_q_heads, sh.head_dim, device="cuda")
        ctx.step(0, trace[t], lay, qd, dl.k, dl.v, out)
        assert ctx.slow_mask() == [int(x) for x in slow_ref[t]]
        if slow_ref[t, 0]:
            idx_g, cnt_g = ctx.selection(0)
            sels[t] = (idx_g.cpu().numpy(), cnt_g.cpu().numpy())
        outs.append(out.cpu().numpy()[0])
    torch.cuda.synchronize()
    assert ctx.read_status() == 0
    ctx.close()
    K64, V64 = dl.K64[0], dl.V64[0]
    held = None
    for t in range(wl.n_steps):
        n = wl.n0[0] + t
        if slow_ref[t, 0]:
            st = O.slow_step(q64s[t], K64, V64, n, wl.n_sink, wl.window, wl.k, wl.lam)
            assert max_abs(outs[t], st["o"]) <= O_TOL["bf16"], t
            idx_g, cnt_g = sels[t]
            for g in range(sh.n_kv_heads):
                check_selection(idx_g[0, g, :cnt_g[0, g]], st["s"][g], st["lo"], st["hi"], wl.k)
            held = [idx_g[0, g, :cnt_g[0, g]].astype(np.int64) for g in range(sh.n_kv_heads)]
        else:
            exp = O.fast_step(q64s[t], K64, V64, n, held, wl.n_sink, wl.window)
            assert max_abs(outs[t], exp) <= O_TOL["bf16"], (t, max_abs(outs[t], exp))


def test_select_top_bin_over_candidate_cap(sfi):
    """More than 8192 keys of E (the candidate list's capacity) share the k-th
    key's top radix digit (the top 11 bits of the fp32 order key), so the
    selector finishes the lower digits with histogram passes over every CTA's
    keys instead of the gathered candidate list.
    KV head 0: 12000 distinct-or-tied scores in one narrow band; KV head 1:
    every score equal (the set is the lowest k positions of E)."""
    ns, win, k = 4, 256, 6000
    n = ns + 12000 + win
    wl = W.small(1, 8, 2, 64, "f32", [n], 21, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, [n])
    ws = sfi.alloc_workspace(lay)
    rng = np.random.default_rng(21)
    f = np.zeros((1, 2, lay.max_len), np.float32)
    u = np.floor(rng.random(n) * 3000.0) / 3000.0  # about four keys per value: exact ties
    f[0, 0, :n] = (1e-4 * (1.0 + 0.1 * u)).astype(np.float32)
    f[0, 1, :n] = np.float32(1.0 / n)
    kn = np.zeros_like(f)
    kn[0, :, :n] = np.float32(2.0)
    prm = sfi.params(ns, win, k, wl.lam)
    idx = torch.full((1, 2, k), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((1, 2), -1, dtype=torch.int32, device="cuda")
    s_out = torch.full((1, 2, lay.max_len), -7.0, device="cuda")
    sfi.sfi_select(lay, prm, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(), idx, cnt, s_out, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    idx, cnt, s_gpu = idx.cpu().numpy(), cnt.cpu().numpy(), s_out.cpu().numpy()
    lo, hi = O.eligible_range(n, ns, win)
    f64, kn64 = f[0, :, :n].astype(np.float64), kn[0, :, :n].astype(np.float64)
    s_ref = O.fuse(f64, O.prior_r(kn64, lo, hi), wl.lam)
    assert max_abs(s_gpu[0, :, :n], s_ref) <= S_TOL
    # the premise: the k-th key's top digit holds more than 8192 keys of E
    for g in range(2):
        keys = s_gpu[0, g, lo:hi].astype(np.float32).view(np.uint32)
        keys = np.where(keys & 0x80000000, ~keys, keys | 0x80000000) >> 21
        kth = np.sort(keys)[::-1][k - 1]
        assert int(np.sum(keys == kth)) > 8192
        sel = idx[0, g, :cnt[0, g]]
        check_selection(sel, s_ref[g], lo, hi, k)
        assert np.array_equal(sel, O.top_k(s_gpu[0, g].astype(np.float64), lo, hi, k))
    assert np.array_equal(idx[0, 1, :k], np.arange(lo, lo + k))


def test_select_ties_across_chunks_within_candidate_cap(sfi):
    """The k-th key's top digit holds most of E but fewer than 8192 keys, and
    E spans several chunk CTAs: the gathered candidate list decides the lower
    digits, and the keys equal to the k-th one that are kept are the lowest-
    positioned ones across chunk boundaries.  KV head 0: 7900 scores in one
    narrow band with about four keys per value; KV head 1: every score equal
    (the set is the lowest k positions of E)."""
    ns, win, k = 4, 256, 3000
    n = ns + 7900 + win
    wl = W.small(1, 8, 2, 64, "f32", [n], 23, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, [n])
    ws = sfi.alloc_workspace(lay)
    rng = np.random.default_rng(23)
    f = np.zeros((1, 2, lay.max_len), np.float32)
    u = np.floor(rng.random(n) * 2000.0) / 2000.0
    f[0, 0, :n] = (1e-4 * (1.0 + 0.1 * u)).astype(np.float32)
    f[0, 1, :n] = np.float32(1.0 / n)
    kn = np.zeros_like(f)
    kn[0, :, :n] = np.float32(2.0)
    prm = sfi.params(ns, win, k, wl.lam)
    idx = torch.full((1, 2, k), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((1, 2), -1, dtype=torch.int32, device="cuda")
    s_out = torch.full((1, 2, lay.max_len), -7.0, device="cuda")
    for rep in range(2):  # the second call finds the counters the first one left
        sfi.sfi_select(lay, prm, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(), idx, cnt, s_out, ws)
        torch.cuda.synchronize()
        assert sfi.sfi_read_status(ws) == 0
        idx_h, cnt_h, s_gpu = idx.cpu().numpy(), cnt.cpu().numpy(), s_out.cpu().numpy()
        lo, hi = O.eligible_range(n, ns, win)
        f64, kn64 = f[0, :, :n].astype(np.float64), kn[0, :, :n].astype(np.float64)
        s_ref = O.fuse(f64, O.prior_r(kn64, lo, hi), wl.lam)
        assert max_abs(s_gpu[0, :, :n], s_ref) <= S_TOL
        for g in range(2):
            keys = s_gpu[0, g, lo:hi].astype(np.float32).view(np.uint32)
            keys = np.where(keys & 0x80000000, ~keys, keys | 0x80000000)
            kth = np.sort(keys)[::-1][k - 1]
            in_bin = int(np.sum((keys >> 21) == (kth >> 21)))
            assert k < in_bin <= 8192  # the premise
            # ties at the k-th key straddle positions beyond one chunk
            assert int(np.sum(keys == kth)) > 1
            sel = idx_h[0, g, :cnt_h[0, g]]
            check_selection(sel, s_ref[g], lo, hi, k)
            assert np.array_equal(sel, O.top_k(s_gpu[0, g].astype(np.float64), lo, hi, k))
        assert np.array_equal(idx_h[0, 1, :k], np.arange(lo, lo + k))


def test_fast_only_launch_short_units(sfi):
    """A launch of fast units only deals each unit's rows over the items of the
    row bound n_sink + k + window; units with far fewer rows (|E| < k, or E
    empty) leave some of their items without rows, and those must weigh
    nothing in the merge.  Lengths 6000, 300 and 40 with k = 1500: 25, 5 and
    1 stages of rows against a bound of 25."""
    B, hq, hkv, d, ns, win, k = 3, 32, 8, 128, 4, 64, 1500
    lens = [6000, 300, 40]
    wl = W.small(B, hq, hkv, d, "bf16", lens, 23, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, q64 = dl.queries(0)
    rng = np.random.default_rng(23)
    idx = np.zeros((B, hkv, k), np.int32)
    cnt = np.zeros((B, hkv), np.int32)
    for b in range(B):
        lo, hi = O.eligible_range(lens[b], ns, win)
        ke = max(0, min(k, hi - lo))
        for g in range(hkv):
            idx[b, g, :ke] = np.sort(rng.choice(np.arange(lo, hi), size=ke, replace=False)) if ke else []
            cnt[b, g] = ke
    out = torch.full((B, hq, d), float("nan"), device="cuda")
    sfi.sfi_fast_attn(lay, sfi.params(ns, win, k, wl.lam), qd, dl.k, dl.v, torch.from_numpy(idx).cuda(),
                      torch.from_numpy(cnt).cuda(), out, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    out = out.cpu().numpy()
    for b in range(B):
        exp = O.fast_step(q64[b], dl.K64[b], dl.V64[b], lens[b],
                          [idx[b, g, :cnt[b, g]].astype(np.int64) for g in range(hkv)], ns, win)
        assert max_abs(out[b], exp) <= O_TOL["bf16"], (b, max_abs(out[b], exp))
