"""The premise of the GPU refinement kernel, checked on the CPU against the
oracle's greedy Soft-NMS (builder's reading of the SFI pages' Selector
section): taking every "local winner" (a remaining position that beats every
remaining position within 2 rho of itself) per round, then applying their
decays, picks the same positions with the same scores as the one-at-a-time
greedy; and the greedy's first k picks lie in the top (k - 1)(4 rho + 1) + 1
positions by starting score, so the rounds may run on those candidates only.
A plain-Python restatement of the kernel's algorithm, not the kernel."""
import math

import numpy as np

import oracle.sfi_oracle as O


def rounds_select(score, lo, hi, k, rho, sigma, n_cand=None):
    """Local-winner rounds on the top-M candidates; the k best picks (ascending)."""
    n_e = hi - lo
    M = min(n_e, (k - 1) * (4 * rho + 1) + 1 if n_cand is None else n_cand)
    pos = np.arange(lo, hi)
    order = np.lexsort((pos, -np.asarray(score[lo:hi], np.float64)))
    cand = np.sort(pos[order[:M]])
    v = {int(p): float(score[p]) for p in cand}
    alive = set(v)
    picked = {}
    reach = 2 * rho

    def beats(a, b):  # a ahead of b: larger score, then lower position
        return v[a] > v[b] or (v[a] == v[b] and a < b)

    while alive:
        win = [i for i in alive
               if not any(j in alive and j != i and beats(j, i) for j in range(i - reach, i + reach + 1))]
        assert win, "the best remaining candidate is always a local winner"
        for i in win:
            picked[i] = v[i]
            alive.discard(i)
        for j in alive:
            for i in win:
                d = abs(i - j)
                if d <= reach:
                    o = O.nms_overlap(d, rho)
                    v[j] *= math.exp(-o * o / sigma)
        best = max((v[j] for j in alive), default=None)
        if best is None or sum(1 for s in picked.values() if s > best) >= min(k, n_e):
            break
    top = sorted(picked, key=lambda i: (-picked[i], i))[:min(k, n_e)]
    return sorted(top), picked


def test_rounds_equal_greedy_on_candidates():
    rng = np.random.default_rng(3)
    for trial in range(150):
        n = int(rng.integers(8, 70))
        rho = int(rng.integers(1, 4))
        sigma = float(rng.uniform(0.05, 3.0))
        lo, hi = int(rng.integers(0, 4)), n - int(rng.integers(0, 4))
        k = int(rng.integers(1, max(2, hi - lo)))
        score = rng.random(n)
        got, picked = rounds_select(score, lo, hi, k, rho, sigma)
        taken, at = O.soft_nms(score, lo, hi, k, rho, sigma)
        assert got == sorted(taken.tolist()), (trial, n, rho, k)
        # each of the greedy's picks carries the same score in the rounds
        for p, s in zip(taken.tolist(), at.tolist()):
            assert math.isclose(picked[p], s, rel_tol=1e-12), (trial, p)


def test_candidate_bound_is_tight():
    """Blocks of 4 rho + 1 positions, each block's centre ahead of the rest of
    its block and every block ahead of the next, under near-hard suppression:
    each pick removes its whole block, so the k-th pick ranks exactly
    (k - 1)(4 rho + 1) + 1 by starting score.  The rounds on that many
    candidates reproduce the greedy; one candidate fewer does not."""
    for rho, k in [(1, 5), (2, 4)]:
        w = 4 * rho + 1
        n = k * w + 3
        score = np.zeros(n)
        for b in range(k):
            base = 10.0 * (k - b)
            score[b * w:(b + 1) * w] = base + 1.0
            score[b * w + 2 * rho] = base + 2.0  # the centre
        score[k * w:] = 0.5
        M = (k - 1) * w + 1
        taken, _ = O.soft_nms(score, 0, n, k, rho, 1e-300)
        got, _ = rounds_select(score, 0, n, k, rho, 1e-300)
        assert got == sorted(taken.tolist()) == [b * w + 2 * rho for b in range(k)]
        short, _ = rounds_select(score, 0, n, k, rho, 1e-300, n_cand=M - 1)
        assert short != got
