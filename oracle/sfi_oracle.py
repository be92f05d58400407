"""fp64 CPU oracle of the SFI decode-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs use it.  It shares no code with the CUDA path;
its inputs come from ``sfi_workloads`` (seeded generators, no method arithmetic).

Sources (web-page summaries of "Slow-Fast Inference: Training-Free Inference
Acceleration via Within-Sentence Support Stability", gist.science paper
2603.12038, in Italian, Portuguese and Korean; and of "Vegas", gist.science
paper 2602.07223, in Italian):

* fast step: attention over sink tokens, a recent sliding window and the
  selected memory only (SFI it/pt/ko pages, section "Slow-Fast paradigm",
  item "Fast Steps");
* slow step: dense full attention over the whole history; its attention logits
  are the evidence (same section, item "Slow Steps");
* selector: evidence distribution f from the slow step's logits, prior r from
  cache statistics (key norms), closed-form reverse-KL fusion
  s = (1-lambda) f + lambda r, then Top-K (SFI ko page, section 2.B "Selector",
  the objective and its closed form);
* Vegas: T = argmax over k-subsets of the prefix of the summed attention logits
  (Vegas page, section 2.A formula), with logits collected from the first draft
  row and the bonus row only (section 2.B "Collect-2-Query").

Readings where the pages leave a step open (each one is listed in the design
notes): f is the softmax probability of the decode row averaged over the query
heads of a KV head; the prior is the key L2 norm normalised over the eligible
set E = [n_sink, n - window); the window includes the current token; ties in
Top-K go to the lower position and the result is returned in ascending
position order; Soft-NMS and cross-head exclusivity (named on the pages without
a formula) are optional refinements in the builder's reading stated at the
end of this module, off unless asked for.

Parity: every function here is pinned by ``tests/test_oracle.py`` against
library routines, closed forms, brute force or hand-computed fixtures; the
end-to-end decode loop is pinned only through its per-step parts.

Notation: n is the cache length including the current token; q is [H_q, d];
K, V are [H_kv, >= n, d]; query head h reads KV head g = h // G, G = H_q / H_kv.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np


# ------------------------------------------------------------------ attention

def attention_over_rows(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                        rows: Sequence[np.ndarray]) -> Tuple[np.ndarray, List[np.ndarray], List[np.ndarray]]:
    """Softmax attention of every query head over the listed cache rows of its KV head.

    ``rows[g]`` lists the positions KV head g attends to.  For query head h
    (KV head g = h // G): l_{h,i} = q_h . k_{g,i} / sqrt(d) for i in rows[g],
    p_h = softmax(l_h), o_h = sum_i p_{h,i} v_{g,i}.
    Returns (o [H_q, d], logits per head, probabilities per head).
    """
    q = np.asarray(q, np.float64)
    hq, d = q.shape
    hkv = K.shape[0]
    G = hq // hkv
    scale = 1.0 / math.sqrt(d)
    o = np.zeros((hq, d))
    logits: List[np.ndarray] = []
    probs: List[np.ndarray] = []
    for h in range(hq):
        g = h // G
        r = np.asarray(rows[g], np.int64)
        if r.size == 0:
            logits.append(np.zeros(0))
            probs.append(np.zeros(0))
            continue
        kk = np.asarray(K[g][r], np.float64)
        vv = np.asarray(V[g][r], np.float64)
        l = (kk @ q[h]) * scale
        e = np.exp(l - l.max())
        p = e / e.sum()
        o[h] = p @ vv
        logits.append(l)
        probs.append(p)
    return o, logits, probs


def dense_attention(q, K, V, n: int):
    """Slow step attention: every head attends to all positions [0, n).

    Returns (o [H_q, d], logits [H_q, n], p [H_q, n]).
    """
    hkv = K.shape[0]
    o, lg, pr = attention_over_rows(q, K, V, [np.arange(n)] * hkv)
    return o, np.stack(lg), np.stack(pr)


# ------------------------------------------------------------------ selector

def evidence_f(p: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """Evidence distribution of each KV head: the mean of its G query heads'
    softmax probabilities.  p [H_q, n] -> f [H_kv, n]; each row sums to 1."""
    hq, n = p.shape
    G = hq // n_kv_heads
    return p.reshape(n_kv_heads, G, n).mean(axis=1)


def eligible_range(n: int, n_sink: int, window: int) -> Tuple[int, int]:
    """Eligible set E = [n_sink, n - window) (empty when n <= n_sink + window).

    Sinks and the recent window are always in the fast set, so selection is
    made only among the positions between them."""
    lo = n_sink
    hi = max(n_sink, n - window)
    return lo, hi


def key_norms(K: np.ndarray, n: int) -> np.ndarray:
    """Cache statistic nu_{g,i} = ||k_{g,i}||_2 for i < n: [H_kv, n]."""
    k = np.asarray(K[:, :n], np.float64)
    return np.sqrt(np.sum(k * k, axis=-1))


def prior_r(nu: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Prior r: key norms normalised over E = [lo, hi), zero elsewhere.
    nu [H_kv, n] -> r [H_kv, n].  With E empty, r is all zero."""
    r = np.zeros_like(nu)
    if hi > lo:
        tot = nu[:, lo:hi].sum(axis=1, keepdims=True)
        r[:, lo:hi] = nu[:, lo:hi] / tot
    return r


def fuse(f: np.ndarray, r: np.ndarray, lam: float) -> np.ndarray:
    """Closed-form reverse-KL fusion: argmin_s (1-lam) KL(f||s) + lam KL(r||s)
    over the simplex is the convex mixture s = (1-lam) f + lam r."""
    return (1.0 - lam) * f + lam * r


def top_k(score: np.ndarray, lo: int, hi: int, k: int) -> np.ndarray:
    """The min(k, |E|) positions of E = [lo, hi) with the largest score.

    Order key (-score_i, i): among equal scores the lower position wins.
    The result is returned in ascending position order."""
    if hi <= lo or k <= 0:
        return np.zeros(0, np.int64)
    pos = np.arange(lo, hi)
    sc = np.asarray(score[lo:hi], np.float64)
    order = np.lexsort((pos, -sc))  # primary: -score, secondary: position
    keep = pos[order[:min(k, hi - lo)]]
    return np.sort(keep)


def slow_step(q, K, V, n: int, n_sink: int, window: int, k: int, lam: float) -> Dict:
    """One slow step of one sequence: dense attention, evidence, prior, fusion, Top-K."""
    hkv = K.shape[0]
    o, logits, p = dense_attention(q, K, V, n)
    f = evidence_f(p, hkv)
    nu = key_norms(K, n)
    lo, hi = eligible_range(n, n_sink, window)
    r = prior_r(nu, lo, hi)
    s = fuse(f, r, lam)
    idx = [top_k(s[g], lo, hi, k) for g in range(hkv)]
    return dict(o=o, logits=logits, p=p, f=f, knorm=nu, r=r, s=s, lo=lo, hi=hi, idx=idx)


# ------------------------------------------------------------------ fast step

def fast_rows(n: int, idx: np.ndarray, n_sink: int, window: int) -> np.ndarray:
    """Fast-step row set: sinks [0, min(n_sink, n)) + selected idx + recent
    window [max(n_sink, n - window), n).  The three parts are disjoint when idx
    was selected from E at an earlier (or the same) length."""
    sinks = np.arange(0, min(n_sink, n))
    win = np.arange(max(n_sink, n - window), n)
    idx = np.asarray(idx, np.int64)
    rows = np.concatenate([sinks, idx, win]).astype(np.int64)
    if np.unique(rows).size != rows.size:
        raise ValueError("fast-step row set is not disjoint")
    return rows


def fast_step(q, K, V, n: int, idx: Sequence[np.ndarray], n_sink: int, window: int):
    """Sparse attention over each KV head's managed state at length n: o [H_q, d]."""
    hkv = K.shape[0]
    rows = [fast_rows(n, idx[g], n_sink, window) for g in range(hkv)]
    o, _, _ = attention_over_rows(q, K, V, rows)
    return o


# ------------------------------------------------------------------ scheduling

def schedule(is_boundary: np.ndarray, budget: int) -> np.ndarray:
    """Slow/fast decision per (step, sequence).

    A sequence runs a slow step at a boundary, when it has no selection yet
    (its first step), or when the fast steps since its last slow step have
    reached ``budget`` (budget 0: unlimited).  Otherwise it runs a fast step.
    is_boundary [T, B] -> slow [T, B] (bool)."""
    T, B = is_boundary.shape
    slow = np.zeros((T, B), bool)
    for b in range(B):
        have_sel = False
        since = 0
        for t in range(T):
            s = bool(is_boundary[t, b]) or not have_sel or (budget > 0 and since >= budget)
            slow[t, b] = s
            if s:
                have_sel = True
                since = 0
            else:
                since += 1
    return slow


def decode_sequence(qs: Sequence[np.ndarray], K, V, n0: int, slow_mask: Sequence[bool],
                    n_sink: int, window: int, k: int, lam: float) -> List[Dict]:
    """Run the slow/fast decode loop of one sequence and one layer.

    Step t runs at length n0 + t with query qs[t]; slow steps refresh the
    selection that later fast steps reuse."""
    out = []
    idx = None
    for t, q in enumerate(qs):
        n = n0 + t
        if slow_mask[t] or idx is None:
            st = slow_step(q, K, V, n, n_sink, window, k, lam)
            idx = st["idx"]
            st["kind"] = "slow"
            st["n"] = n
            out.append(st)
        else:
            o = fast_step(q, K, V, n, idx, n_sink, window)
            out.append(dict(kind="fast", o=o, n=n, idx=idx))
    return out


# ------------------------------------------------------------------ Vegas

def verify_attention(q_rows: np.ndarray, K, V, n_pre: int):
    """Verification attention with R = gamma + 1 query rows.

    Row t sits at position n_pre + t and attends to [0, n_pre + t] (the prefix
    plus a causal tail).  q_rows [R, H_q, d] -> (o [R, H_q, d],
    logits[t] [H_q, n_pre + t + 1])."""
    R = q_rows.shape[0]
    o = np.zeros(q_rows.shape)
    logits = []
    for t in range(R):
        o[t], lg, _ = dense_attention(q_rows[t], K, V, n_pre + t + 1)
        logits.append(lg)
    return o, logits


def collected_logit_sum(logits: Sequence[np.ndarray], rows: Sequence[int], n_pre: int,
                        n_kv_heads: int = 1) -> np.ndarray:
    """L_i = sum over collected rows t and query heads h of l^{(h)}_{t,i}, i in
    the prefix P = [0, n_pre).  With n_kv_heads > 1 the sum is kept per KV
    head (over that head's query group): [n_kv_heads, n_pre]."""
    hq = logits[0].shape[0]
    G = hq // n_kv_heads
    L = np.zeros((n_kv_heads, n_pre))
    for t in rows:
        lg = logits[t][:, :n_pre]
        L += lg.reshape(n_kv_heads, G, n_pre).sum(axis=1)
    return L


def vegas_select(L: np.ndarray, k: int) -> np.ndarray:
    """T = argmax over k-subsets of the prefix of sum_{i in T} L_i: the top-k of
    L (ties to the lower position), in ascending order."""
    return top_k(L, 0, L.shape[0], k)


def draft_rows(n_pre: int, n: int, T: np.ndarray) -> np.ndarray:
    """Draft-step rows at length n: the selected prefix set T plus every position
    since the prefix, [n_pre, n)."""
    return np.concatenate([np.asarray(T, np.int64), np.arange(n_pre, n)])


def draft_step(q, K, V, n_pre: int, n: int, T: np.ndarray):
    hkv = K.shape[0]
    rows = [draft_rows(n_pre, n, T)] * hkv
    o, _, _ = attention_over_rows(q, K, V, rows)
    return o


# ------------------------------------------------------------------ selector refinements
#
# The SFI pages list two refinements of the selector beside the fusion: a
# Soft-NMS that keeps one head from spending its budget on neighbouring,
# correlated tokens, and a cross-head exclusivity that penalises a token
# chosen again by another head (it/pt/ko pages, section "Selector").  They
# give no formula for either, so these functions are the builder's reading:
#
# * Soft-NMS is the greedy Gaussian-decay Soft-NMS of Bodla et al. (ICCV
#   2017) with position i of E treated as the 1-D box [i - rho, i + rho]:
#   repeatedly take the largest current score (ties to the lower position);
#   every remaining position j whose box overlaps the taken one (|i - j| <=
#   2 rho) has its score multiplied by exp(-IoU(i, j)^2 / sigma).  The first
#   min(k, |E|) positions taken are the selection.  rho = 0 is plain Top-K.
# * Exclusivity: the KV heads of a sequence select in index order; head g's
#   fused scores are multiplied by exp(-beta * c_i), where c_i counts the
#   heads before g whose selection holds i.  beta = 0 is no exclusivity.

def nms_overlap(d: int, rho: int) -> float:
    """Intersection over union of the position boxes [i - rho, i + rho] and
    [j - rho, j + rho] at distance d = |i - j| (0 once they no longer meet)."""
    w = 2 * rho + 1
    return max(0, w - d) / (w + d)


def soft_nms(score: np.ndarray, lo: int, hi: int, k: int, rho: int, sigma: float):
    """Greedy Soft-NMS over E = [lo, hi): the first min(k, |E|) positions taken,
    in the order taken, and each one's score at the moment it was taken."""
    if hi <= lo or k <= 0:
        return np.zeros(0, np.int64), np.zeros(0)
    v = np.array(score[lo:hi], np.float64)
    alive = np.ones(hi - lo, bool)
    taken, at = [], []
    for _ in range(min(k, hi - lo)):
        i = int(np.argmax(np.where(alive, v, -np.inf)))  # first maximum: lower position
        taken.append(lo + i)
        at.append(v[i])
        alive[i] = False
        for j in range(max(0, i - 2 * rho), min(hi - lo, i + 2 * rho + 1)):
            if alive[j]:
                o = nms_overlap(abs(i - j), rho)
                v[j] *= math.exp(-o * o / sigma)
    return np.array(taken, np.int64), np.array(at)


def refine_head(s_g: np.ndarray, counts: np.ndarray, lo: int, hi: int, k: int, rho: int,
                sigma: float, beta: float):
    """Selection of one KV head given the counts of earlier heads' picks.

    Returns (ascending positions, each position's score when it was taken,
    in the same order)."""
    sh = np.asarray(s_g, np.float64) * np.exp(-beta * np.asarray(counts, np.float64))
    if rho > 0:
        taken, at = soft_nms(sh, lo, hi, k, rho, sigma)
    else:
        taken = top_k(sh, lo, hi, k)
        at = sh[taken]
    order = np.argsort(taken)
    return taken[order], at[order]


def refined_select(s: np.ndarray, lo: int, hi: int, k: int, rho: int, sigma: float,
                   beta: float) -> List[np.ndarray]:
    """Selections of every KV head of one sequence (s [H_kv, n]), heads in
    index order, with exclusivity (beta) and Soft-NMS (rho, sigma)."""
    counts = np.zeros(s.shape[1])
    out = []
    for g in range(s.shape[0]):
        idx, _ = refine_head(s[g], counts, lo, hi, k, rho, sigma, beta)
        counts[idx] += 1
        out.append(idx)
    return out
