"""Full-size parity: the batch-8, 131072-context decode in the launch
configuration the benchmark times (one mixed slow/fast launch per layer,
cache filled on the device), checked on sampled (layer, sequence) units
against the fp64 oracle fed with the same inputs regenerated on the CPU."""
import numpy as np
import pytest
import torch

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import O_TOL, check_selection, load_sfi, max_abs

pytestmark = pytest.mark.gpu

SAMPLES = [(1, 3), (0, 6)]  # (layer, sequence)
STEPS = 40


def test_cfg2_decode_sampled_units():
    assert torch.cuda.is_available()
    sfi = load_sfi()
    import bench
    wl = W.cfg2(n_layers=2, n_steps=STEPS)
    R = bench.Cfg2Runner(wl, 0)
    sh = wl.shape
    # record the outputs of every (step, layer) for the sampled units
    outs = {}
    for t in range(wl.n_steps):
        lay = R.layouts[t]
        for l in range(wl.n_layers):
            r = sfi.lib.sfi_decode_step(R.ctx.h, l, R.bnd[t], lay, R.Q[l][t].data_ptr(), R.kp[l],
                                        R.vp[l], R.op[l], R.stream.cuda_stream)
            assert r == 0
            masks = R.ctx.slow_mask()
            for (sl, sb) in SAMPLES:
                if sl == l:
                    outs[(t, l, sb)] = R.out[l][sb].clone()
                    if masks[sb]:  # refreshed: keep the set the next fast steps use
                        outs[("sel", t, l, sb)] = R.ctx.selection(l)
        if t == 0:
            mask0 = R.ctx.slow_mask()
        outs[("mask", t)] = R.ctx.slow_mask()
    torch.cuda.synchronize()
    assert mask0 == [1] * sh.batch  # first step: no selection yet
    trace = wl.boundary_trace()
    slow_ref = O.schedule(trace, wl.budget)
    for t in range(wl.n_steps):
        assert outs[("mask", t)] == [int(x) for x in slow_ref[t]], t
    for (l, b) in SAMPLES:
        cap = wl.cap[b]
        # inputs of this unit, regenerated on the CPU; they must equal the device bytes
        k_st = wl.kv_storage("k", l, b)
        v_st = wl.kv_storage("v", l, b)
        per = sh.n_kv_heads * cap * sh.head_dim
        kd = R.K[l][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        vd = R.V[l][R.offsets[b]:R.offsets[b] + per].view(torch.int16).cpu().numpy().view(np.uint16)
        # the two generators may differ only where the fp64 math libraries
        # round differently at a bf16 rounding boundary (~1e-13 per element)
        assert int(np.sum(kd != k_st.reshape(-1))) <= 2 and int(np.sum(vd != v_st.reshape(-1))) <= 2
        # the oracle reads the CPU generator's values only
        K64 = W.storage_to_f64(k_st, "bf16")
        V64 = W.storage_to_f64(v_st, "bf16")
        qs = []
        for t in range(wl.n_steps):
            q_st = wl.q_storage(l, t, b)
            qd = R.Q[l][t][b].view(torch.int16).cpu().numpy().view(np.uint16)
            assert int(np.sum(qd != q_st)) <= 1
            qs.append(W.storage_to_f64(q_st, "bf16"))
        ref = O.decode_sequence(qs, K64, V64, wl.n0[b], slow_ref[:, b], wl.n_sink, wl.window,
                                wl.k, wl.lam)
        gsel = None
        for t in range(wl.n_steps):
            got = outs[(t, l, b)].cpu().numpy()
            if ref[t]["kind"] == "slow":
                exp = ref[t]["o"]
                idx_g, cnt_g = outs[("sel", t, l, b)]
                idx_g, cnt_g = idx_g.cpu().numpy()[b], cnt_g.cpu().numpy()[b]
                st = ref[t]
                for g in range(sh.n_kv_heads):
                    check_selection(idx_g[g, :cnt_g[g]], st["s"][g], st["lo"], st["hi"], wl.k)
                gsel = [idx_g[g, :cnt_g[g]].astype(np.int64) for g in range(sh.n_kv_heads)]
            else:
                # the fast step with the set the GPU selected at the last refresh
                exp = O.fast_step(qs[t], K64, V64, wl.n0[b] + t, gsel, wl.n_sink, wl.window)
            err = max_abs(got, exp)
            assert err <= O_TOL["bf16"], (l, b, t, ref[t]["kind"], err)
