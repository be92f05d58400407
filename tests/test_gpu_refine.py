"""GPU parity of the selector refinements -- Soft-NMS within a KV head and
cross-head exclusivity, in the builder's reading of the SFI pages' Selector
section -- against the fp64 oracle, through the C ABI (binding).

Decisions inside the greedy are taken in fp32 on the GPU and in fp64 in the
oracle; the oracle is run on the GPU's own fused scores s, and each KV head's
exclusivity counts come from the GPU's selections of the earlier heads, so a
difference at a near-tie of one head cannot spread to the next.  The sets
must agree except at positions whose score at the pick lies within 1e-6
(relative) of the k-th pick's."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import DeviceLayer, S_TOL, TIE_RTOL, load_sfi, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sfi():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return load_sfi()


def run_refined(sfi, lay, prm, ref, f_d, kn_d, B, hkv, k):
    ws = torch.zeros(sfi.select_refined_workspace_size(lay, prm, ref), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    idx = torch.full((B, hkv, k), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, hkv), -1, dtype=torch.int32, device="cuda")
    s = torch.full((B, hkv, lay.max_len), -7.0, device="cuda")
    sfi.sfi_select_refined(lay, prm, ref, f_d, kn_d, idx, cnt, s, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    return idx.cpu().numpy(), cnt.cpu().numpy(), s.cpu().numpy()


def check_refined(idx, cnt, s_gpu, n, lo, hi, k, rho, sigma, beta):
    """One sequence: every KV head's set against the oracle's greedy."""
    hkv = s_gpu.shape[0]
    counts = np.zeros(s_gpu.shape[1])
    ke = max(0, min(k, hi - lo))
    for g in range(hkv):
        got = idx[g, :cnt[g]]
        assert cnt[g] == ke, (g, cnt[g], ke)
        if ke == 0:
            continue
        assert np.all(np.diff(got) > 0), "selection not strictly ascending"
        assert got.min() >= lo and got.max() < hi, "selection outside E"
        extra = min(hi - lo, k + 32)
        sg = s_gpu[g].astype(np.float64)
        sg[n:] = 0.0
        ox, at = O.refine_head(sg, counts, lo, hi, extra, rho, sigma, beta)
        order = np.lexsort((ox, -at))  # pick order: scores at the pick never increase
        first = ox[order[:ke]]
        tau = at[order[ke - 1]]
        amb = {int(i) for i, a in zip(ox, at) if abs(a - tau) <= TIE_RTOL * abs(tau)}
        bad = [i for i in set(got.tolist()) ^ set(first.tolist()) if i not in amb]
        assert not bad, f"head {g}: {len(bad)} non-ambiguous positions differ, e.g. {sorted(bad)[:6]}"
        counts[got] += 1


# (B, H_q, H_kv, d, dtype, lens, n_sink, window, k, seed)
SMALL = [
    (2, 8, 2, 64, "f32", [2048, 1500], 4, 256, 128, 11),
    (3, 16, 4, 128, "bf16", [3000, 700, 300], 4, 64, 200, 12),  # third: M > |E| > k
    (2, 8, 4, 64, "f32", [40, 300], 4, 16, 50, 13),             # first: |E| <= k, all of E
    (2, 8, 2, 64, "f32", [10, 600], 4, 16, 8, 14),              # first: E empty
    (1, 8, 2, 64, "f32", [60], 4, 16, 8, 15),  # 40 candidates: slices of 5 < 2 rho (rho = 8)
]
REFINES = [(1, 0.5, 0.0), (2, 0.3, 0.7), (0, 1.0, 1.5), (4, 2.0, 0.2), (8, 0.1, 0.0)]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}-hkv{c[2]}-{c[4]}-k{c[8]}")
def test_refined_selection_parity(sfi, case):
    B, hq, hkv, d, dt, lens, ns, win, k, seed = case
    wl = W.small(B, hq, hkv, d, dt, lens, seed, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, q64 = dl.queries(0)
    out = torch.empty(B, hq, d, device="cuda")
    f_d = torch.zeros(B, hkv, lay.max_len, device="cuda")
    kn_d = torch.zeros_like(f_d)
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, f_d, kn_d, ws)
    torch.cuda.synchronize()
    assert sfi.sfi_read_status(ws) == 0
    prm = sfi.params(ns, win, k, wl.lam)
    # plain selection, for the no-refinement identity
    idx0 = torch.full((B, hkv, k), -1, dtype=torch.int32, device="cuda")
    cnt0 = torch.full((B, hkv), -1, dtype=torch.int32, device="cuda")
    sfi.sfi_select(lay, prm, f_d, kn_d, idx0, cnt0, None, ws)
    torch.cuda.synchronize()
    idx0, cnt0 = idx0.cpu().numpy(), cnt0.cpu().numpy()
    for rho, sigma, beta in REFINES + [(0, 1.0, 0.0)]:
        ref = sfi.sfi_refine(rho, sigma, beta)
        idx, cnt, s = run_refined(sfi, lay, prm, ref, f_d, kn_d, B, hkv, k)
        if rho == 0 and beta == 0.0:
            np.testing.assert_array_equal(cnt, cnt0)
            for b in range(B):
                for g in range(hkv):
                    np.testing.assert_array_equal(idx[b, g, :cnt[b, g]], idx0[b, g, :cnt0[b, g]])
            continue
        for b in range(B):
            n = lens[b]
            st = O.slow_step(q64[b], dl.K64[b], dl.V64[b], n, ns, win, k, wl.lam)
            assert max_abs(s[b, :, :n], st["s"]) <= S_TOL
            assert np.all(s[b, :, n:] == -7.0), "wrote past n"
            check_refined(idx[b], cnt[b], s[b], n, st["lo"], st["hi"], k, rho, sigma, beta)
        # the same call again gives the same bytes
        idx2, cnt2, _ = run_refined(sfi, lay, prm, ref, f_d, kn_d, B, hkv, k)
        np.testing.assert_array_equal(cnt2, cnt)
        np.testing.assert_array_equal(idx2, idx)


def synthetic_evidence(B, hkv, n_max, lens, seed):
    """Seeded stand-ins for f and the key norms at full context: per (b, g), 1%
    of the positions carry a heavy logit; f is the softmax; norms ~ |N(0, I_128)|."""
    rng = np.random.default_rng(seed)
    f = np.zeros((B, hkv, n_max), np.float32)
    kn = np.zeros((B, hkv, n_max), np.float32)
    for b in range(B):
        n = lens[b]
        for g in range(hkv):
            lg = 0.8 * rng.standard_normal(n)
            lg[rng.choice(n, n // 100, replace=False)] += 4.0
            e = np.exp(lg - lg.max())
            f[b, g, :n] = e / e.sum()
            kn[b, g, :n] = np.sqrt(rng.chisquare(128, n))
    return f, kn


@pytest.mark.parametrize("refine", [(1, 0.5, 0.5), (2, 0.3, 0.0)], ids=["rho1-excl", "rho2"])
def test_refined_selection_full_context(sfi, refine):
    """Two sequences at 131072 and 100000 positions, 8 KV heads, k = 4096,
    window 256: rho = 1 (20476 candidates per unit) with exclusivity, and
    rho = 2 (36856 candidates per unit)."""
    B, hkv, k, ns, win, lam = 2, 8, 4096, 4, 256, 0.3
    lens = [131072, 100000]
    n_max = 131072
    f, kn = synthetic_evidence(B, hkv, n_max, lens, 21)
    lay = sfi.Layout(32, hkv, 128, torch.bfloat16, [0, 0], [n_max, n_max], lens, n_max)
    prm = sfi.params(ns, win, k, lam)
    rho, sigma, beta = refine
    ref = sfi.sfi_refine(rho, sigma, beta)
    idx, cnt, s = run_refined(sfi, lay, prm, ref, torch.from_numpy(f).cuda(), torch.from_numpy(kn).cuda(),
                              B, hkv, k)
    for b in range(B):
        n = lens[b]
        lo, hi = O.eligible_range(n, ns, win)
        f64 = f[b, :, :n].astype(np.float64)
        r = O.prior_r(kn[b, :, :n].astype(np.float64), lo, hi)
        assert max_abs(s[b, :, :n], O.fuse(f64, r, lam)) <= S_TOL
        check_refined(idx[b], cnt[b], s[b], n, lo, hi, k, rho, sigma, beta)
    # Soft-NMS spreads the picks: fewer adjacent pairs than the plain Top-K
    plain = O.top_k(s[0, 0].astype(np.float64), *O.eligible_range(lens[0], ns, win), k)
    assert np.sum(np.diff(idx[0, 0, :k]) <= 2) < np.sum(np.diff(plain) <= 2)


@pytest.mark.parametrize("refine", [(2, 0.3, 0.5), (1, 0.5, 0.0)], ids=["nms2-excl", "nms1"])
def test_decode_driver_refined(sfi, refine):
    """The decode driver with a refinement: two layers, an all-slow step, a fast
    step, then a mixed step (sequence 1 at a boundary).  The in-line and the
    overlapped selector give the same bytes; every refreshed set matches the
    oracle's refined selection, every output the oracle's attention (fast
    steps over the sets the GPU held)."""
    B, hq, hkv, d, ns, win, k = 2, 8, 4, 64, 4, 64, 40
    lens = [900, 1300]
    wl = W.small(B, hq, hkv, d, "f32", lens, 31, n_sink=ns, window=win, k=k, n_steps=4)
    dl = DeviceLayer.build(wl)
    prm = sfi.params(ns, win, k, wl.lam)
    rho, sigma, beta = refine
    bnd = [[0, 0], [0, 0], [0, 1]]
    runs = {}
    for async_select in (False, True):
        ctx = sfi.DecodeContext(B, hq, hkv, d, torch.float32, max(wl.cap), 2, prm, 0,
                                async_select=async_select, refine=sfi.sfi_refine(rho, sigma, beta))
        lay = dl.layout(sfi, lens)
        outs, sels, masks = [], [], []
        for t in range(3):
            lay.set_lens([n + t for n in lens])
            qd, _ = dl.queries(t)
            o_t = []
            for layer in range(2):
                out = torch.empty(B, hq, d, device="cuda")
                ctx.step(layer, bnd[t], lay, qd, dl.k, dl.v, out)
                o_t.append(out)
            masks.append(ctx.slow_mask())
            sel = [tuple(x.cpu().numpy() for x in ctx.selection(layer)) for layer in range(2)]
            outs.append([o.cpu().numpy() for o in o_t])
            sels.append(sel)
        torch.cuda.synchronize()
        assert ctx.read_status() == 0
        ctx.close()
        runs[async_select] = (outs, sels, masks)
    (o0, s0, m0), (o1, s1, m1) = runs[False], runs[True]
    assert m0 == m1 == [[1, 1], [0, 0], [0, 1]]
    for t in range(3):
        for layer in range(2):
            np.testing.assert_array_equal(o0[t][layer], o1[t][layer])
            for a, b in zip(s0[t][layer], s1[t][layer]):
                np.testing.assert_array_equal(a, b)
    held = {}
    for t in range(3):
        n_t = [n + t for n in lens]
        _, q64 = dl.queries(t)
        for b in range(B):
            for layer in range(2):
                idx, cnt = s0[t][layer]
                if m0[t][b]:
                    st = O.slow_step(q64[b], dl.K64[b], dl.V64[b], n_t[b], ns, win, k, wl.lam)
                    assert max_abs(o0[t][layer][b], st["o"]) <= 2e-5
                    check_refined(idx[b], cnt[b], st["s"], n_t[b], st["lo"], st["hi"], k, rho, sigma, beta)
                    held[(b, layer)] = [idx[b, g, :cnt[b, g]].astype(np.int64) for g in range(hkv)]
                else:
                    ref = O.fast_step(q64[b], dl.K64[b], dl.V64[b], n_t[b], held[(b, layer)], ns, win)
                    assert max_abs(o0[t][layer][b], ref) <= 2e-5


# Relative near-tie band of the chained comparison.  The GPU's fused scores
# carry the fp32 error of logits accumulated over head_dim products (about
# 1e-6 relative near the selection boundary, checked below against a quarter
# of the band) and fp32 decay factors (about 1e-7).
CHAIN_EPS = 1e-5


def chain_allowance(sh_or, c_or, c_gpu, lo, hi, k, rho, sigma, eps):
    """Positions where the oracle's chain and the GPU's may legitimately differ
    for one KV head: (1) picks whose score at the pick lies within eps of the
    k-th pick's (the set boundary); (2) interacting neighbours (|i - j| <= 2 rho)
    whose starting scores are within eps of each other (the greedy may take
    either first); (3) positions whose exclusivity count differs between the
    two chains (earlier heads differed there).  Each with its 2 rho neighbours."""
    ext = min(hi - lo, k + 64)
    if rho > 0:
        taken, at = O.soft_nms(sh_or, lo, hi, ext, rho, sigma)
    else:
        taken = O.top_k(sh_or, lo, hi, ext)
        taken = taken[np.lexsort((taken, -sh_or[taken]))]
        at = sh_or[taken]
    tau = at[min(k, hi - lo) - 1]
    seeds = set(int(i) for i, a in zip(taken, at) if abs(a - tau) <= eps * abs(tau))
    e = sh_or[lo:hi]
    for d in range(1, 2 * rho + 1):
        close = np.abs(e[d:] - e[:-d]) <= eps * np.maximum(e[d:], e[:-d])
        for i in np.nonzero(close)[0]:
            seeds.update((lo + int(i), lo + int(i) + d))
    seeds.update(int(i) for i in np.nonzero(c_or != c_gpu)[0])
    allowed = set()
    for i in seeds:
        allowed.update(range(i - 2 * rho, i + 2 * rho + 1))
    return allowed


@pytest.mark.parametrize("refine", [(1, 0.5, 0.0), (2, 0.3, 0.5)], ids=["nms1", "nms2-excl"])
def test_refined_chain_vs_oracle_chain(sfi, refine):
    """What a user of the refined selection gets, end to end: the GPU's slow
    step -> f and key norms -> refined selection, against the oracle's own
    chain (slow step -> refined selection in fp64), with nothing from the GPU
    fed to the oracle.  The sets may differ only inside the stated near-tie
    band (chain_allowance), and by at most 1% of k per KV head."""
    B, hq, hkv, d, ns, win, k = 2, 32, 8, 128, 4, 256, 1024
    lens = [20000, 13001]
    wl = W.small(B, hq, hkv, d, "bf16", lens, 61, n_sink=ns, window=win, k=k)
    dl = DeviceLayer.build(wl)
    lay = dl.layout(sfi, lens)
    ws = sfi.alloc_workspace(lay)
    qd, q64 = dl.queries(0)
    out = torch.empty(B, hq, d, device="cuda")
    f_d = torch.zeros(B, hkv, lay.max_len, device="cuda")
    kn_d = torch.zeros_like(f_d)
    sfi.sfi_slow_attn(lay, qd, dl.k, dl.v, out, f_d, kn_d, ws)
    prm = sfi.params(ns, win, k, wl.lam)
    rho, sigma, beta = refine
    idx, cnt, s_gpu = run_refined(sfi, lay, prm, sfi.sfi_refine(rho, sigma, beta), f_d, kn_d, B, hkv, k)
    for b in range(B):
        n = lens[b]
        st = O.slow_step(q64[b], dl.K64[b], dl.V64[b], n, ns, win, k, wl.lam)
        lo, hi = st["lo"], st["hi"]
        s_or = st["s"]
        sets_or = O.refined_select(s_or, lo, hi, k, rho, sigma, beta)
        c_or = np.zeros(n)
        c_gpu = np.zeros(n)
        for g in range(hkv):
            got = idx[b, g, :cnt[b, g]].astype(np.int64)
            exp = sets_or[g]
            assert len(got) == len(exp) == min(k, hi - lo)
            sh_or = s_or[g] * np.exp(-beta * c_or)
            # the premise of the band: the GPU's scores are within it where it matters
            top = sh_or[lo:hi] >= 0.1 * np.sort(sh_or[lo:hi])[::-1][len(exp) - 1]
            rel = np.abs(s_gpu[b, g, lo:hi] - s_or[g, lo:hi]) / s_or[g, lo:hi]
            assert float(rel[top].max()) <= 0.25 * CHAIN_EPS
            diff = set(got.tolist()) ^ set(exp.tolist())
            allowed = chain_allowance(sh_or, c_or, c_gpu, lo, hi, k, rho, sigma, CHAIN_EPS)
            outside = sorted(diff - allowed)
            assert not outside, f"seq {b} head {g}: {len(outside)} positions differ outside the band: {outside[:6]}"
            assert len(diff) <= max(4, k // 100), (b, g, len(diff))
            c_or[exp] += 1
            c_gpu[got] += 1
