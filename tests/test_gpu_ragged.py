"""Ragged serving batch: 32 sequences with contexts log-uniform in
[4096, 262144], bf16, Llama-3-8B attention shape.  An all-slow step at n - 1
builds every selection; the next step mixes 8 slow and 24 fast sequences in one
launch.  Sampled sequences (the two shortest of each kind) are checked against
the fp64 oracle at every (k, window) point of the sweep."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import O_TOL, check_selection, load_sfi, max_abs

pytestmark = pytest.mark.gpu

POINTS = [(1024, 128), (4096, 256), (16384, 512), (16384, 128)]


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
    samples = sorted(slow_set, key=lambda b: lens[b])[:2] + sorted(fast_set, key=lambda b: lens[b])[:2]
    # inputs of the sampled sequences, regenerated on the CPU (must match the device bytes)
    inp = {}
    for b in samples:
        k_st = base.kv_storage("k", 0, b)
        v_st = base.kv_storage("v", 0, b)
        per = sh.n_kv_heads * base.cap[b] * sh.head_dim
        kd = R.K[0][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        vd = R.V[0][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        assert int(np.sum(kd != k_st.reshape(-1))) <= 2 and int(np.sum(vd != v_st.reshape(-1))) <= 2
        q = []
        for t in range(2):
            q_st = base.q_storage(0, t, b)
            qd = R.Q[0][t][b].view(torch.int16).cpu().numpy().view(np.uint16)
            assert int(np.sum(qd != q_st)) <= 1
            q.append(W.storage_to_f64(q_st, "bf16"))
        # the oracle reads the CPU generator's values only
        inp[b] = (W.storage_to_f64(k_st, "bf16"), W.storage_to_f64(v_st, "bf16"), q)
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
        idx0, cnt0 = (x.cpu().numpy() for x in sel0)
        for b in samples:
            K64, V64, q = inp[b]
            n = lens[b]
            st0 = O.slow_step(q[0], K64, V64, n - 1, base.n_sink, win, k, base.lam)
            assert max_abs(out0[b].cpu().numpy(), st0["o"]) <= O_TOL["bf16"]
            for g in range(sh.n_kv_heads):
                check_selection(idx0[b, g, :cnt0[b, g]], st0["s"][g], st0["lo"], st0["hi"], k)
            if b in slow_set:
                exp = O.slow_step(q[1], K64, V64, n, base.n_sink, win, k, base.lam)["o"]
            else:
                gsel = [idx0[b, g, :cnt0[b, g]].astype(np.int64) for g in range(sh.n_kv_heads)]
                exp = O.fast_step(q[1], K64, V64, n, gsel, base.n_sink, win)
            assert max_abs(out1[b].cpu().numpy(), exp) <= O_TOL["bf16"], (k, win, b)
        ctx.close()
