"""Planted mistakes in the oracle must be caught by its pins.

Each case patches one oracle function (on the CPU, in this process only) with a
plausible mistake: a dropped term, a wrong sign or index, an off-by-one, a
transposed operand.  The test passes when at least one pin of
``test_oracle.py`` fails on the mutated oracle.
"""
import math

import numpy as np
import pytest

import oracle.sfi_oracle as O
import tests.test_oracle as P

ALL_PINS = [getattr(P, n) for n in dir(P) if n.startswith("pin_")]


def _attn_wrong_group(q, K, V, rows):
    # query head h reads KV head h % H_kv instead of h // G
    hq, d = q.shape
    hkv = K.shape[0]
    o = np.zeros((hq, d)); lg = []; pr = []
    for h in range(hq):
        g = h % hkv
        r = np.asarray(rows[g], np.int64)
        l = (K[g][r] @ q[h]) / math.sqrt(d)
        e = np.exp(l - l.max()); p = e / e.sum()
        o[h] = p @ V[g][r]; lg.append(l); pr.append(p)
    return o, lg, pr


def _attn_no_scale(q, K, V, rows):
    hq, d = q.shape
    G = hq // K.shape[0]
    o = np.zeros((hq, d)); lg = []; pr = []
    for h in range(hq):
        g = h // G
        r = np.asarray(rows[g], np.int64)
        l = K[g][r] @ q[h]
        e = np.exp(l - l.max()); p = e / e.sum()
        o[h] = p @ V[g][r]; lg.append(l); pr.append(p)
    return o, lg, pr


def _attn_uses_k_for_v(q, K, V, rows):
    return O.__dict__["_orig_attention_over_rows"](q, K, K, rows)


MUTANTS = {
    "fusion weights swapped": ("fuse", lambda f, r, lam: lam * f + (1 - lam) * r),
    "fusion drops prior": ("fuse", lambda f, r, lam: (1 - lam) * f),
    "evidence sums instead of mean": ("evidence_f", lambda p, hkv: p.reshape(hkv, -1, p.shape[1]).sum(1)),
    "evidence takes first head only": ("evidence_f", lambda p, hkv: p.reshape(hkv, -1, p.shape[1])[:, 0]),
    "attention wrong GQA group": ("attention_over_rows", _attn_wrong_group),
    "attention missing 1/sqrt(d)": ("attention_over_rows", _attn_no_scale),
    "attention reads K as V": ("attention_over_rows", _attn_uses_k_for_v),
    "window excludes current token": ("eligible_range", lambda n, ns, w: (ns, max(ns, n - w + 1))),
    "eligible set includes sinks": ("eligible_range", lambda n, ns, w: (0, max(ns, n - w))),
    "norm squared": ("key_norms", lambda K, n: np.sum(np.asarray(K[:, :n]) ** 2, axis=-1)),
    "prior over all positions": ("prior_r", lambda nu, lo, hi: nu / nu.sum(1, keepdims=True)),
    "top-k ties to higher position": ("top_k", lambda s, lo, hi, k: np.sort(
        np.arange(lo, hi)[np.lexsort((-np.arange(lo, hi), -np.asarray(s[lo:hi])))[:min(k, max(0, hi - lo))]])
        if hi > lo and k > 0 else np.zeros(0, np.int64)),
    "top-k smallest": ("top_k", lambda s, lo, hi, k: np.sort(
        np.arange(lo, hi)[np.lexsort((np.arange(lo, hi), np.asarray(s[lo:hi])))[:min(k, max(0, hi - lo))]])
        if hi > lo and k > 0 else np.zeros(0, np.int64)),
    "fast window off by one": ("fast_rows", lambda n, idx, ns, w: np.concatenate(
        [np.arange(0, min(ns, n)), np.asarray(idx, np.int64), np.arange(max(ns, n - w - 1), n)])),
    "schedule budget strict": ("schedule", None),
    "collect uses rows 0 and 1": ("collected_logit_sum", None),
    "verify without causal tail": ("verify_attention", None),
    "soft-nms IoU without the distance in the union": ("nms_overlap", lambda d, rho: max(0, 2 * rho + 1 - d) / (2 * rho + 1)),
    "soft-nms reaches only rho": ("soft_nms", None),
    "soft-nms decay with IoU not squared": ("soft_nms", None),
    "soft-nms ties to higher position": ("soft_nms", None),
    "exclusivity rewards repeated picks": ("refine_head", None),
    "exclusivity ignores earlier heads": ("refined_select", None),
}


def _schedule_strict(is_boundary, budget):
    T, B = is_boundary.shape
    slow = np.zeros((T, B), bool)
    for b in range(B):
        have, since = False, 0
        for t in range(T):
            s = bool(is_boundary[t, b]) or not have or (budget > 0 and since > budget)
            slow[t, b] = s
            have, since = (True, 0) if s else (have, since + 1)
    return slow


def _collect_rows01(logits, rows, n_pre, n_kv_heads=1):
    return O.__dict__["_orig_collected_logit_sum"](logits, [0, 1], n_pre, n_kv_heads)


def _verify_no_tail(q_rows, K, V, n_pre):
    R = q_rows.shape[0]
    o = np.zeros(q_rows.shape); logits = []
    for t in range(R):
        o[t], lg, _ = O.dense_attention(q_rows[t], K, V, n_pre)
        logits.append(np.concatenate([lg, np.zeros((lg.shape[0], t + 1))], axis=1))
    return o, logits


def _soft_nms_variant(reach, power, last_max):
    def run(score, lo, hi, k, rho, sigma):
        if hi <= lo or k <= 0:
            return np.zeros(0, np.int64), np.zeros(0)
        v = np.array(score[lo:hi], np.float64)
        alive = np.ones(hi - lo, bool)
        taken, at = [], []
        for _ in range(min(k, hi - lo)):
            cur = np.where(alive, v, -np.inf)
            i = int(len(cur) - 1 - np.argmax(cur[::-1])) if last_max else int(np.argmax(cur))
            taken.append(lo + i); at.append(v[i]); alive[i] = False
            r = reach(rho)
            for j in range(max(0, i - r), min(hi - lo, i + r + 1)):
                if alive[j]:
                    o = O.nms_overlap(abs(i - j), rho)
                    v[j] *= math.exp(-o ** power / sigma)
        return np.array(taken, np.int64), np.array(at)
    return run


def _refine_head_reward(s_g, counts, lo, hi, k, rho, sigma, beta):
    return O.__dict__["_orig_refine_head"](s_g, counts, lo, hi, k, rho, sigma, -beta)


def _refined_select_no_counts(s, lo, hi, k, rho, sigma, beta):
    return [O.refine_head(s[g], np.zeros(s.shape[1]), lo, hi, k, rho, sigma, beta)[0]
            for g in range(s.shape[0])]


SPECIAL = {"schedule budget strict": _schedule_strict,
           "collect uses rows 0 and 1": _collect_rows01,
           "verify without causal tail": _verify_no_tail,
           "soft-nms reaches only rho": _soft_nms_variant(lambda r: r, 2, False),
           "soft-nms decay with IoU not squared": _soft_nms_variant(lambda r: 2 * r, 1, False),
           "soft-nms ties to higher position": _soft_nms_variant(lambda r: 2 * r, 2, True),
           "exclusivity rewards repeated picks": _refine_head_reward,
           "exclusivity ignores earlier heads": _refined_select_no_counts}


def _caught(monkeypatch) -> bool:
    for pin in ALL_PINS:
        try:
            pin(O)
        except Exception:
            return True
    return False


def test_unmutated_oracle_passes_all_pins():
    for pin in ALL_PINS:
        pin(O)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    fn_name, repl = MUTANTS[name]
    if repl is None:
        repl = SPECIAL[name]
    monkeypatch.setitem(O.__dict__, "_orig_" + fn_name, getattr(O, fn_name))
    monkeypatch.setattr(O, fn_name, repl)
    assert _caught(monkeypatch), f"planted mistake '{name}' passed every pin"
