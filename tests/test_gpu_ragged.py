"""Ragged serving batch: 32 sequences with contexts log-uniform in
[4096, 262144], bf16, Llama-3-8B attention shape.  An all-slow step at n - 1
builds every selection; the next step mixes 8 slow and 24 fast sequences in one
launch.  At every (k, window) point of the sweep -- k in {1024, 4096, 16384} x
window in {128, 256, 512} -- the shortest and the longest sequences of each
kind (contexts from 4323 to 231752) are checked against the fp64 oracle: the dense outputs, every KV
head's selection (tie rule) and the fast outputs over the sets the GPU held."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import O_TOL, check_selection, load_sfi, max_abs

pytestmark = pytest.mark.gpu

POINTS = [(k, w) for k in (1024, 4096, 16384) for w in (128, 256, 512)]


def test_ragged_mixed_step():
    assert torch.cuda.is_available()
    sfi = load_sfi()
    import bench
    import ctypes
    base = W.cfg4()
    R = bench.Cfg2Runner(base, 0)
    sh = base.shape
    lens = [n + 1 for n in base.n0]
    slow_set = [int(x) for x in W.cfg4_slow_set()]
    fast_set = [b for b in range(sh.batch) if b not in slow_set]
    by_len = lambda bs: sorted(bs, key=lambda b: lens[b])
    # the two shortest and two longest slow sequences; the two shortest and the
    # four longest fast ones (118281 to 231752 positions)
    samples = (by_len(slow_set)[:2] + by_len(slow_set)[-2:] + by_len(fast_set)[:2] +
               by_len(fast_set)[-4:])
    # Inputs of the sampled sequences, regenerated on the CPU (they must match
    # the device bytes); the oracle reads the CPU generator's values only.  The
    # dense attention of each sampled sequence at n - 1 (and at n for the slow
    # ones) does not depend on (k, window): it is computed once, and each sweep
    # point applies the oracle's prior, fusion and Top-K to it -- the slow
    # step's own composition (pinned against O.slow_step below).
    ref = {}
    for b in samples:
        k_st = base.kv_storage("k", 0, b)
        v_st = base.kv_storage("v", 0, b)
        per = sh.n_kv_heads * base.cap[b] * sh.head_dim
        kd = R.K[0][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        vd = R.V[0][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        assert int(np.sum(kd != k_st.reshape(-1))) <= 2 and int(np.sum(vd != v_st.reshape(-1))) <= 2
        del kd, vd
        q = []
        for t in range(2):
            q_st = base.q_storage(0, t, b)
            qd = R.Q[0][t][b].view(torch.int16).cpu().numpy().view(np.uint16)
            assert int(np.sum(qd != q_st)) <= 1
            q.append(W.storage_to_f64(q_st, "bf16"))
        K64, V64 = W.storage_to_f64(k_st, "bf16"), W.storage_to_f64(v_st, "bf16")
        del k_st, v_st
        n = lens[b]
        o0, _, p0 = O.dense_attention(q[0], K64, V64, n - 1)
        f0 = O.evidence_f(p0, sh.n_kv_heads)
        del p0
        nu0 = O.key_norms(K64, n - 1)
        o1 = O.dense_attention(q[1], K64, V64, n)[0] if b in slow_set else None
        if b == samples[0]:
            # the per-point composition is the oracle's slow step
            st = O.slow_step(q[0], K64, V64, n - 1, base.n_sink, 256, 4096, base.lam)
            lo, hi = O.eligible_range(n - 1, base.n_sink, 256)
            s_c = O.fuse(f0, O.prior_r(nu0, lo, hi), base.lam)
            assert np.array_equal(s_c, st["s"]) and np.array_equal(o0, st["o"])
            del st
        if b in slow_set:  # only the fast sequences' rows are read again
            K64 = V64 = None
        ref[b] = dict(K64=K64, V64=V64, q1=q[1], o0=o0, f0=f0, nu0=nu0, o1=o1)

    bnd1 = (ctypes.c_uint8 * sh.batch)(*[1 if b in slow_set else 0 for b in range(sh.batch)])
    for k, win in POINTS:
        ctx = sfi.DecodeContext(sh.batch, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, torch.bfloat16,
                                R.max_len, 1, sfi.params(base.n_sink, win, k, base.lam), 0)
        assert sfi.lib.sfi_decode_step(ctx.h, 0, R.bnd[0], R.layouts[0], R.Q[0][0].data_ptr(), R.kp[0],
                                       R.vp[0], R.op[0], R.stream.cuda_stream) == 0
        out0 = R.out[0].clone()
        sel0 = ctx.selection(0)
        assert sfi.lib.sfi_decode_step(ctx.h, 0, bnd1, R.layouts[1], R.Q[0][1].data_ptr(), R.kp[0],
                                       R.vp[0], R.op[0], R.stream.cuda_stream) == 0
        out1 = R.out[0].clone()
        torch.cuda.synchronize()
        assert ctx.slow_mask() == [1 if b in slow_set else 0 for b in range(sh.batch)]
        assert ctx.read_status() == 0
        idx0, cnt0 = (x.cpu().numpy() for x in sel0)
        for b in samples:
            r = ref[b]
            n = lens[b]
            assert max_abs(out0[b].cpu().numpy(), r["o0"]) <= O_TOL["bf16"], (k, win, b)
            lo, hi = O.eligible_range(n - 1, base.n_sink, win)
            s = O.fuse(r["f0"], O.prior_r(r["nu0"], lo, hi), base.lam)
            for g in range(sh.n_kv_heads):
                check_selection(idx0[b, g, :cnt0[b, g]], s[g], lo, hi, k)
            if b in slow_set:
                exp = r["o1"]
            else:
                gsel = [idx0[b, g, :cnt0[b, g]].astype(np.int64) for g in range(sh.n_kv_heads)]
                exp = O.fast_step(r["q1"], r["K64"], r["V64"], n, gsel, base.n_sink, win)
            assert max_abs(out1[b].cpu().numpy(), exp) <= O_TOL["bf16"], (k, win, b)
        ctx.close()
