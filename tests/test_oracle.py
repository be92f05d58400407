"""Pins of the fp64 oracle against things other than itself.

Each pin checks the oracle against a library routine (torch's fp64
scaled_dot_product_attention, scipy's constrained minimiser), a closed form, a
hand-computed fixture under tests/golden/ (each citing the passage it follows),
brute-force enumeration on tiny inputs, or an invariant the method fixes.
``test_oracle_mutations.py`` plants mistakes in the oracle and checks that
these pins catch them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def sdpa(q, K, V, n, mask=None):
    """torch fp64 SDPA with the KV heads repeated for their query groups."""
    hq, d = q.shape
    hkv = K.shape[0]
    G = hq // hkv
    qt = torch.tensor(q)[None, :, None, :]
    kt = torch.tensor(K[:, :n]).repeat_interleave(G, dim=0)[None]
    vt = torch.tensor(V[:, :n]).repeat_interleave(G, dim=0)[None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)[0, :, 0].numpy()


# ---------------------------------------------------------------- attention

def pin_dense_vs_sdpa(O):
    for seed, (hq, hkv, d, n) in enumerate([(8, 2, 16, 37), (4, 4, 8, 5), (6, 1, 32, 64), (32, 8, 128, 300)]):
        q, K, V = rnd(seed, hq, d), rnd(seed + 100, hkv, n + 3, d), rnd(seed + 200, hkv, n + 3, d)
        o, logits, p = O.dense_attention(q, K, V, n)
        np.testing.assert_allclose(o, sdpa(q, K, V, n), atol=1e-12, rtol=0)
        # probabilities: SDPA with V = identity returns the softmax matrix itself
        eye = np.broadcast_to(np.eye(n)[None], (hkv, n, n)).copy()
        np.testing.assert_allclose(p, sdpa(q, K, eye, n), atol=1e-13, rtol=0)
        np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-12)


def test_dense_attention_matches_sdpa():
    pin_dense_vs_sdpa(O)


def pin_attention_hand(O):
    g = gold("attention_hand.json")
    o, logits, p = O.dense_attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]), 3)
    np.testing.assert_allclose(p, g["p"], atol=1e-15)
    np.testing.assert_allclose(o, g["o"], atol=1e-14)


def test_attention_hand_fixture():
    pin_attention_hand(O)


# ---------------------------------------------------------------- evidence

def pin_evidence(O):
    hq, hkv, d, n = 8, 2, 16, 50
    q, K, V = rnd(1, hq, d), rnd(2, hkv, n, d), rnd(3, hkv, n, d)
    _, _, p = O.dense_attention(q, K, V, n)
    f = O.evidence_f(p, hkv)
    np.testing.assert_allclose(f.sum(1), 1.0, atol=1e-12)
    assert (f >= 0).all()
    eye = np.broadcast_to(np.eye(n)[None], (hkv, n, n)).copy()
    P = sdpa(q, K, eye, n)  # [hq, n] from the library
    G = hq // hkv
    for g in range(hkv):
        np.testing.assert_allclose(f[g], P[g * G:(g + 1) * G].mean(0), atol=1e-13)


def test_evidence_is_group_mean_of_softmax():
    pin_evidence(O)


# ---------------------------------------------------------------- prior / fusion

def pin_fusion_hand(O):
    g = gold("fusion_hand.json")
    K = np.array(g["k_rows"])[None]
    nu = O.key_norms(K, g["n"])
    np.testing.assert_allclose(nu[0], g["knorm"], atol=0)
    lo, hi = O.eligible_range(g["n"], g["n_sink"], g["window"])
    r = O.prior_r(nu, lo, hi)
    np.testing.assert_allclose(r[0], g["r"], atol=1e-15)
    s = O.fuse(np.array(g["f"])[None], r, g["lam"])
    np.testing.assert_allclose(s[0], g["s"], atol=1e-15)
    assert list(O.top_k(s[0], lo, hi, 1)) == g["top1"]
    assert list(O.top_k(s[0], lo, hi, 2)) == g["top2"]
    assert list(O.top_k(s[0], lo, hi, 5)) == g["top5"]


def test_fusion_hand_fixture():
    pin_fusion_hand(O)


def pin_knorm_closed_form(O):
    # rows c_i * (unit vector) have norm |c_i|; Pythagorean triples
    K = np.zeros((2, 5, 6))
    K[0, 0, :2] = [3, 4]; K[0, 1, 2:4] = [5, 12]; K[0, 2, 5] = -7; K[0, 3, :3] = [2, 3, 6]
    K[1, :, 0] = [1, 2, 3, 4, 5]
    nu = O.key_norms(K, 4)
    np.testing.assert_allclose(nu, [[5, 13, 7, 7], [1, 2, 3, 4]], atol=1e-15)


def test_key_norm_closed_form():
    pin_knorm_closed_form(O)


def pin_prior(O):
    nu = np.abs(rnd(5, 3, 40)) + 0.1
    for (lo, hi) in [(4, 30), (0, 40), (10, 11)]:
        r = O.prior_r(nu, lo, hi)
        np.testing.assert_allclose(r[:, lo:hi].sum(1), 1.0, atol=1e-14)
        assert (r[:, :lo] == 0).all() and (r[:, hi:] == 0).all()
        # proportional to the norm inside E
        np.testing.assert_allclose(r[:, lo:hi] * nu[:, lo:hi].sum(1, keepdims=True), nu[:, lo:hi], rtol=1e-13)
    assert (O.prior_r(nu, 7, 7) == 0).all()


def test_prior_normalised_on_eligible_set():
    pin_prior(O)


def kl(a, b):
    m = a > 0
    return float(np.sum(a[m] * np.log(a[m] / b[m])))


def pin_fusion_objective(O):
    """The closed form is the minimiser of (1-lam) KL(f||s) + lam KL(r||s) on the simplex."""
    from scipy.optimize import minimize
    rng = np.random.default_rng(7)
    for lam in [0.0, 0.3, 0.5, 0.9, 1.0]:
        n = 12
        f = rng.dirichlet(np.ones(n))
        r = np.zeros(n)
        r[2:9] = rng.dirichlet(np.ones(7))
        s = O.fuse(f[None], r[None], lam)[0]
        np.testing.assert_allclose(s.sum(), 1.0, atol=1e-14)
        if lam == 0.0:
            np.testing.assert_array_equal(s, f)
        if lam == 1.0:
            np.testing.assert_array_equal(s, r)

        def obj(x):
            z = np.exp(x - x.max())
            sv = z / z.sum()
            return (1 - lam) * kl(f, sv) + lam * kl(r, sv)

        x0 = np.zeros(n)
        res = minimize(obj, x0, method="L-BFGS-B", options=dict(ftol=1e-15, gtol=1e-12, maxiter=5000))
        z = np.exp(res.x - res.x.max())
        s_num = z / z.sum()
        np.testing.assert_allclose(s_num, s, atol=2e-4)
        assert obj(np.log(np.maximum(s, 1e-300))) <= res.fun + 1e-9
        # stationarity on the simplex: ((1-lam) f_i + lam r_i) / s_i = 1 where s_i > 0
        m = s > 0
        np.testing.assert_allclose(((1 - lam) * f[m] + lam * r[m]) / s[m], 1.0, atol=1e-13)


def test_fusion_minimises_reverse_kl_objective():
    pin_fusion_objective(O)


# ---------------------------------------------------------------- top-k

def brute_best(score, cand, k):
    best, arg = -math.inf, []
    for sub in itertools.combinations(cand, k):
        v = float(sum(score[i] for i in sub))
        if v > best + 1e-12:
            best, arg = v, [sub]
        elif abs(v - best) <= 1e-12:
            arg.append(sub)
    return best, arg


def pin_topk_bruteforce(O):
    rng = np.random.default_rng(11)
    for trial in range(40):
        n = int(rng.integers(3, 13))
        lo = int(rng.integers(0, 3))
        hi = int(rng.integers(lo, n + 1))
        s = rng.random(n)
        for k in range(0, hi - lo + 2):
            got = O.top_k(s, lo, hi, k)
            ke = min(k, hi - lo)
            assert len(got) == ke
            assert list(got) == sorted(got)
            if ke == 0:
                continue
            _, arg = brute_best(s, range(lo, hi), ke)
            assert tuple(got) in [tuple(sorted(a)) for a in arg]


def test_topk_is_best_subset_by_enumeration():
    pin_topk_bruteforce(O)


def pin_topk_ties(O):
    s = np.array([0.5, 0.2, 0.2, 0.2, 0.9, 0.2, 0.1])
    assert list(O.top_k(s, 0, 7, 3)) == [0, 1, 4]
    assert list(O.top_k(s, 2, 7, 2)) == [2, 4]
    assert list(O.top_k(np.zeros(6), 1, 6, 2)) == [1, 2]
    assert list(O.top_k(s, 3, 3, 5)) == []
    assert list(O.top_k(s, 1, 4, 10)) == [1, 2, 3]


def test_topk_ties_go_to_lower_position():
    pin_topk_ties(O)


# ---------------------------------------------------------------- sets / schedule

def pin_sets_hand(O):
    for c in gold("sets_hand.json")["cases"]:
        assert list(O.eligible_range(c["n"], c["n_sink"], c["window"])) == c["E"]
        assert list(O.fast_rows(c["n"], np.array(c["idx"], np.int64), c["n_sink"], c["window"])) == c["rows"]


def test_sets_hand_fixture():
    pin_sets_hand(O)


def pin_schedule_hand(O):
    g = gold("schedule_hand.json")
    b = np.array(g["is_boundary"], np.uint8)[:, None]
    assert list(O.schedule(b, g["budget"])[:, 0].astype(int)) == g["slow"]
    assert list(O.schedule(b, 0)[:, 0].astype(int)) == g["budget0_slow"]


def test_schedule_hand_trace():
    pin_schedule_hand(O)


# ---------------------------------------------------------------- fast step

def pin_fast_all_equals_dense(O):
    """With k >= |E| the fast step at the slow step's length is dense attention."""
    for (hq, hkv, d, n, ns, w) in [(8, 2, 16, 60, 4, 8), (4, 1, 8, 9, 2, 3), (6, 3, 32, 40, 0, 0), (4, 2, 8, 5, 4, 4)]:
        q, K, V = rnd(n, hq, d), rnd(n + 1, hkv, n, d), rnd(n + 2, hkv, n, d)
        st = O.slow_step(q, K, V, n, ns, w, k=n, lam=0.3)
        of = O.fast_step(q, K, V, n, st["idx"], ns, w)
        np.testing.assert_allclose(of, st["o"], atol=1e-12)


def test_fast_step_with_all_positions_is_dense():
    pin_fast_all_equals_dense(O)


def pin_fast_gather_vs_sdpa(O):
    """With no sinks and no window the fast step is attention over the gathered rows."""
    hq, hkv, d, n = 8, 2, 16, 80
    q, K, V = rnd(21, hq, d), rnd(22, hkv, n, d), rnd(23, hkv, n, d)
    idx = [np.array([3, 10, 11, 40, 77]), np.array([0, 1, 2, 60])]
    of = O.fast_step(q, K, V, n, idx, 0, 0)
    G = hq // hkv
    for g in range(hkv):
        Kg, Vg = K[g:g + 1, idx[g]], V[g:g + 1, idx[g]]
        ref = sdpa(q[g * G:(g + 1) * G], Kg, Vg, len(idx[g]))
        np.testing.assert_allclose(of[g * G:(g + 1) * G], ref, atol=1e-12)


def test_fast_step_is_attention_over_gathered_rows():
    pin_fast_gather_vs_sdpa(O)


def pin_fast_window_slides(O):
    """After m fast steps the window has moved by m; positions that slid out and
    were not selected are no longer attended."""
    hq, hkv, d, n = 4, 1, 8, 30
    q, K, V = rnd(31, hq, d), rnd(32, hkv, n + 5, d), rnd(33, hkv, n + 5, d)
    idx = [np.array([6, 9])]
    o = O.fast_step(q, K, V, n + 3, idx, 2, 5)
    rows = np.array([0, 1, 6, 9, 28, 29, 30, 31, 32])
    ref = sdpa(q, K[:, rows], V[:, rows], len(rows))
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_fast_window_slides():
    pin_fast_window_slides(O)


# ---------------------------------------------------------------- Vegas

def pin_verify_causal_vs_sdpa(O):
    R, hq, hkv, d, n_pre = 5, 8, 2, 16, 40
    qr, K, V = rnd(41, R, hq, d), rnd(42, hkv, n_pre + R, d), rnd(43, hkv, n_pre + R, d)
    o, logits = O.verify_attention(qr, K, V, n_pre)
    G = hq // hkv
    n = n_pre + R
    for t in range(R):
        mask = torch.zeros(1, 1, 1, n, dtype=torch.bool)
        mask[..., : n_pre + t + 1] = True
        ref = sdpa(qr[t], K, V, n, mask=mask)
        np.testing.assert_allclose(o[t], ref, atol=1e-12)
        assert logits[t].shape == (hq, n_pre + t + 1)
        for h in range(hq):
            np.testing.assert_allclose(logits[t][h], K[h // G, : n_pre + t + 1] @ qr[t, h] / math.sqrt(d), atol=1e-12)


def test_verify_attention_is_causal_sdpa():
    pin_verify_causal_vs_sdpa(O)


def pin_collect2(O):
    """Collect-2 sums the first and the bonus row only, over all query heads."""
    R, hq, n_pre = 5, 4, 10
    rng = np.random.default_rng(51)
    logits = [rng.standard_normal((hq, n_pre + t + 1)) for t in range(R)]
    L = O.collected_logit_sum(logits, [0, R - 1], n_pre)[0]
    want = sum(logits[t][h, i] for t in (0, R - 1) for h in range(hq) for i in [0])
    np.testing.assert_allclose(L[0], want, atol=1e-12)
    exp = np.zeros(n_pre)
    for t in (0, R - 1):
        for h in range(hq):
            for i in range(n_pre):
                exp[i] += logits[t][h, i]
    np.testing.assert_allclose(L, exp, atol=1e-12)
    # per-KV-head partial sums add up to the total
    Lg = O.collected_logit_sum(logits, [0, R - 1], n_pre, n_kv_heads=2)
    np.testing.assert_allclose(Lg.sum(0), L, atol=1e-12)
    # a middle row must not contribute: make row 1 decisive and check it is ignored
    logits[1][:, 3] += 1e6
    L2 = O.collected_logit_sum(logits, [0, R - 1], n_pre)[0]
    np.testing.assert_allclose(L2, L, atol=1e-9)


def test_collect2_sums_first_and_bonus_rows():
    pin_collect2(O)


def pin_vegas_argmax(O):
    rng = np.random.default_rng(61)
    for trial in range(30):
        n = int(rng.integers(4, 12))
        k = int(rng.integers(1, n + 1))
        L = rng.standard_normal(n) * 3
        T = O.vegas_select(L, k)
        _, arg = brute_best(L, range(n), k)
        assert tuple(T) in [tuple(sorted(a)) for a in arg]


def test_vegas_selection_is_argmax_subset():
    pin_vegas_argmax(O)


def pin_draft_rows(O):
    assert list(O.draft_rows(10, 13, np.array([2, 5]))) == [2, 5, 10, 11, 12]
    assert list(O.draft_rows(10, 10, np.array([1]))) == [1]


def test_draft_rows():
    pin_draft_rows(O)


# ---------------------------------------------------------------- decode loop

def test_decode_loop_uses_refreshed_selection():
    hq, hkv, d, n0, T = 4, 2, 8, 40, 6
    K, V = rnd(71, hkv, n0 + T, d), rnd(72, hkv, n0 + T, d)
    qs = [rnd(80 + t, hq, d) for t in range(T)]
    mask = [True, False, False, True, False, False]
    out = O.decode_sequence(qs, K, V, n0, mask, 2, 5, 4, 0.3)
    assert [o["kind"] for o in out] == ["slow", "fast", "fast", "slow", "fast", "fast"]
    st3 = O.slow_step(qs[3], K, V, n0 + 3, 2, 5, 4, 0.3)
    for g in range(hkv):
        assert list(out[4]["idx"][g]) == list(st3["idx"][g])
    np.testing.assert_allclose(out[5]["o"], O.fast_step(qs[5], K, V, n0 + 5, st3["idx"], 2, 5), atol=0)


# ---------------------------------------------------------------- generator

def test_generator_vectors():
    g = gold("generator_vectors.json")
    assert W.mix64_int(W.PHI) == int(g["splitmix64_state0_first"], 16)
    for x, bits in g["bf16"]:
        assert int(W.f32_to_bf16_bits(np.array([x], np.float32))[0]) == int(bits, 16)


def test_normal_generator_moments_and_ranges():
    z = W.normal_f64(W.stream_key(1, 2, 3), 0, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1) < 0.01
    assert abs(np.mean(z ** 3)) < 0.03 and abs(np.mean(z ** 4) - 3) < 0.06
    # random access: a sub-range equals the slice of the whole
    np.testing.assert_array_equal(W.normal_f64(W.stream_key(1, 2, 3), 1001, 77), z[1001:1078])


def test_workload_recipe():
    wl = W.cfg0()
    u = wl.u_vec(0)
    np.testing.assert_allclose(np.linalg.norm(u), 1.0, atol=1e-15)
    hp = wl.heavy_positions(0, 0)
    assert len(hp) == round(0.01 * wl.cap[0]) and len(np.unique(hp)) == len(hp)
    k = wl.kv_f64("k", 0, 0, 1, 0, wl.cap[0])
    kz = W.normal_f64(wl.key(W.T_K, 0, 0), wl.cap[0] * wl.shape.head_dim, wl.cap[0] * wl.shape.head_dim)
    diff = k - kz.reshape(k.shape)
    np.testing.assert_allclose(diff[hp], np.broadcast_to(3 * u, (len(hp), len(u))), atol=1e-12)
    mask = np.ones(wl.cap[0], bool); mask[hp] = False
    assert np.all(diff[mask] == 0)
    q = wl.q_f64(0, 3, 0)
    assert q.shape == (8, 64)
    tr = W.cfg2().boundary_trace()
    assert tr.shape == (256, 8) and 0.02 < tr.mean() < 0.09


# ------------------------------------------------- selector refinements (builder's reading)

def pin_refine_hand_fixture(O):
    g = gold("refine_hand.json")
    for c in g["soft_nms"]:
        sc = np.array(c["score"])
        for kk in (2, 3, 4):
            if f"k{kk}_taken" not in c:
                continue
            taken, at = O.soft_nms(sc, c["lo"], c["hi"], kk, c["rho"], c["sigma"])
            assert taken.tolist() == c[f"k{kk}_taken"]
            np.testing.assert_allclose(at, c[f"k{kk}_at"], atol=5e-8, rtol=0)
        if "plain_top3" in c:
            assert O.top_k(sc, c["lo"], c["hi"], 3).tolist() == c["plain_top3"]
    for c in g["exclusivity"]:
        s = np.array(c["s"])
        got = O.refined_select(s, c["lo"], c["hi"], c["k"], 0, 1.0, c["beta"])
        assert [x.tolist() for x in got] == c["idx"]
        got0 = O.refined_select(s, c["lo"], c["hi"], c["k"], 0, 1.0, 0.0)
        assert [x.tolist() for x in got0] == c["idx_beta0"]


def test_refine_hand_fixture():
    pin_refine_hand_fixture(O)


def pin_refine_without_refinement_is_topk(O):
    """rho = 0 (or an infinitely wide decay) and beta = 0 leave plain Top-K."""
    rng = np.random.default_rng(7)
    for n, k in [(40, 7), (25, 25), (30, 40)]:
        s = rng.random((3, n))
        for rho, sigma in [(0, 1.0), (2, math.inf)]:
            got = O.refined_select(s, 3, n - 4, k, rho, sigma, 0.0)
            for g in range(3):
                assert got[g].tolist() == O.top_k(s[g], 3, n - 4, k).tolist()


def test_refine_without_refinement_is_topk():
    pin_refine_without_refinement_is_topk(O)


def _hard_nms_by_enumeration(sc, lo, hi, k, rho):
    """Among k-subsets of [lo, hi) whose positions are pairwise more than
    2 rho apart (boxes that do not overlap), the one whose scores, sorted
    from the largest, are lexicographically largest -- what greedy hard
    suppression keeps (the greedy choice on an independence system)."""
    best, best_key = None, None
    for sub in itertools.combinations(range(lo, hi), k):
        if any(b - a <= 2 * rho for a, b in zip(sub, sub[1:])):
            continue
        key = sorted((sc[i] for i in sub), reverse=True)
        if best_key is None or key > best_key:
            best, best_key = list(sub), key
    return best


def pin_soft_nms_hard_limit_by_enumeration(O):
    """As sigma -> 0 every overlapping neighbour of a taken position drops to
    zero, i.e. hard NMS; with enough room for k separated picks the result is
    the enumerated best separated subset."""
    rng = np.random.default_rng(11)
    for rho, k, n in [(1, 3, 12), (2, 2, 12), (1, 2, 9)]:
        for _ in range(6):
            sc = rng.random(n) + 0.01
            taken, _ = O.soft_nms(sc, 0, n, k, rho, 1e-300)
            assert sorted(taken.tolist()) == _hard_nms_by_enumeration(sc, 0, n, k, rho)


def test_soft_nms_hard_limit_by_enumeration():
    pin_soft_nms_hard_limit_by_enumeration(O)


def pin_soft_nms_greedy_trace(O):
    """Each pick is the best remaining position at that moment: its score at
    the pick equals its fused score times the decays of the earlier picks
    within 2 rho, and no remaining position then scores higher (ties: the
    lower position first)."""
    rng = np.random.default_rng(5)
    for rho, sigma in [(1, 0.3), (2, 1.5), (3, 0.05)]:
        n = 60
        sc = rng.random(n)
        taken, at = O.soft_nms(sc, 4, n, 25, rho, sigma)
        assert len(set(taken.tolist())) == 25 and taken.min() >= 4 and taken.max() < n

        def current(j, before):
            x = sc[j]
            for p in before:
                d = abs(p - j)
                if d <= 2 * rho:
                    iou = (2 * rho + 1 - d) / (2 * rho + 1 + d)
                    x *= math.exp(-iou * iou / sigma)
            return x

        for t, p in enumerate(taken):
            before = taken[:t].tolist()
            assert math.isclose(at[t], current(p, before), rel_tol=1e-12)
            for j in range(4, n):
                if j == p or j in before:
                    continue
                cj = current(j, before)
                assert cj < at[t] or (cj == at[t] and j > p)
        assert np.all(np.diff(at) <= 1e-15)  # scores at the pick never increase


def test_soft_nms_greedy_trace():
    pin_soft_nms_greedy_trace(O)


def pin_exclusivity_limit_disjoint(O):
    """With an overwhelming beta a position taken by an earlier head is never
    taken again while enough untaken positions remain: head g's set is the
    Top-K of its scores with the earlier heads' picks removed."""
    rng = np.random.default_rng(13)
    s = rng.random((4, 80)) + 0.01
    got = O.refined_select(s, 2, 70, 10, 0, 1.0, 1e6)
    seen = np.zeros(80, bool)
    for g in range(4):
        masked = np.where(seen, 0.0, s[g])
        assert got[g].tolist() == O.top_k(masked, 2, 70, 10).tolist()
        assert not seen[got[g]].any()
        seen[got[g]] = True


def test_exclusivity_limit_disjoint():
    pin_exclusivity_limit_disjoint(O)
