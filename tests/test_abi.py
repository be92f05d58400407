"""CPU checks of the C ABI: the library loads, exports every function that
include/sfi.h declares, and rejects bad arguments on the host before any GPU
work; the host-only schedule step matches the oracle's schedule."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle.sfi_oracle as O
import sfi_workloads as W
from tests.sfi_testlib import ROOT, load_sfi

HEADER = os.path.join(ROOT, "include", "sfi.h")


@pytest.fixture(scope="module")
def sfi():
    return load_sfi()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(sfi_[a-z0-9_]+)\s*\(",
                                 txt, flags=re.M)))


def test_header_declares_the_path_entry_points():
    names = declared_functions()
    for n in ["sfi_slow_attn", "sfi_select", "sfi_fast_attn", "sfi_decode_step"]:
        assert n in names


def test_library_exports_every_declared_function(sfi):
    lib = ctypes.CDLL(sfi.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sfi.h but not exported"
        assert name in sfi.EXPORTS, f"{name} has no binding"
    assert set(sfi.EXPORTS) == set(declared_functions())


FAKE = 0x10000  # never dereferenced: every call below fails host validation first


def layout(sfi, **kw):
    d = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, dtype=sfi.SFI_F32, max_len=100,
             kv_offset=FAKE, kv_cap=FAKE, len=FAKE)
    d.update(kw)
    return sfi.sfi_layout(**d)


def slow(sfi, L, ws=FAKE, ws_bytes=1 << 40, q=FAKE):
    return sfi.lib.sfi_slow_attn(ctypes.byref(L), q, FAKE, FAKE, FAKE, None, None, ws, ws_bytes, None)


def test_host_validation_codes(sfi):
    assert sfi.lib.sfi_slow_attn(None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 40, None) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi, head_dim=96)) == sfi.SFI_ERR_UNSUPPORTED
    assert slow(sfi, layout(sfi, dtype=7)) == sfi.SFI_ERR_UNSUPPORTED
    assert slow(sfi, layout(sfi, n_q_heads=12, n_kv_heads=4)) == sfi.SFI_ERR_UNSUPPORTED  # G = 3
    assert slow(sfi, layout(sfi, n_q_heads=7)) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi, batch=0)) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi, batch=5000)) == sfi.SFI_ERR_CAPACITY
    assert slow(sfi, layout(sfi, batch=1000, n_q_heads=64, n_kv_heads=8)) == sfi.SFI_ERR_CAPACITY
    assert slow(sfi, layout(sfi, max_len=0)) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi, len=None)) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi), q=None) == sfi.SFI_ERR_INVALID_ARG
    assert slow(sfi, layout(sfi), ws=None) == sfi.SFI_ERR_WORKSPACE
    assert slow(sfi, layout(sfi), ws_bytes=16) == sfi.SFI_ERR_WORKSPACE
    assert slow(sfi, layout(sfi), ws=FAKE + 8) == sfi.SFI_ERR_WORKSPACE  # misaligned
    assert "workspace" in sfi.lib.sfi_last_error().decode()


def test_workspace_size_grows_with_geometry(sfi):
    small = sfi.lib.sfi_slow_attn_workspace_size(ctypes.byref(layout(sfi)))
    big = sfi.lib.sfi_slow_attn_workspace_size(ctypes.byref(layout(sfi, max_len=10000)))
    assert 0 < small < big
    assert sfi.lib.sfi_slow_attn_workspace_size(ctypes.byref(layout(sfi, head_dim=3))) == 0


def test_select_and_fast_param_validation(sfi):
    L = layout(sfi)
    def sel(p, ev=FAKE, kn=FAKE):
        return sfi.lib.sfi_select(ctypes.byref(L), ctypes.byref(p), ev, kn, FAKE, FAKE, None, FAKE, 1 << 40, None)
    def fast(p):
        return sfi.lib.sfi_fast_attn(ctypes.byref(L), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert sel(sfi.params(4, 16, 0, 0.3)) == sfi.SFI_ERR_INVALID_ARG        # k = 0
    assert sel(sfi.params(-1, 16, 8, 0.3)) == sfi.SFI_ERR_INVALID_ARG
    assert sel(sfi.params(4, 16, 8, 1.5)) == sfi.SFI_ERR_INVALID_ARG        # lambda outside [0, 1]
    assert sel(sfi.params(4, 16, 8, float("nan"))) == sfi.SFI_ERR_INVALID_ARG
    assert sel(sfi.params(4, 16, 8, 0.3, mode=9)) == sfi.SFI_ERR_INVALID_ARG
    for m in (sfi.SFI_SELECT_LOGIT_SUM_SEQ, sfi.SFI_SELECT_LOGIT_SUM_HEAD):
        assert sel(sfi.params(0, 5, 8, 0.3, mode=m)) == sfi.SFI_ERR_INVALID_ARG  # lambda must be 0
        assert sel(sfi.params(4, 5, 8, 0.0, mode=m)) == sfi.SFI_ERR_INVALID_ARG  # n_sink must be 0
    assert sel(sfi.params(4, 16, 8, 0.3, mode=sfi.SFI_SELECT_LOGIT_SUM_SEQ)) == sfi.SFI_ERR_INVALID_ARG
    assert sel(sfi.params(4, 16, 8, 0.3), kn=None) == sfi.SFI_ERR_INVALID_ARG
    assert sel(sfi.params(4, 16, 8, 0.3), ev=None) == sfi.SFI_ERR_INVALID_ARG
    assert fast(sfi.params(0, 0, 8, 0.3)) == sfi.SFI_ERR_INVALID_ARG        # empty fast set
    assert sfi.lib.sfi_fast_attn(ctypes.byref(L), ctypes.byref(sfi.params(4, 16, 8, 0.3)), FAKE, FAKE, FAKE,
                                 None, FAKE, FAKE, FAKE, 1 << 40, None) == sfi.SFI_ERR_INVALID_ARG


def test_ctx_and_decode_validation(sfi):
    h = ctypes.c_void_p()
    desc = sfi.sfi_ctx_desc(2, 8, 2, 64, sfi.SFI_F32, 100, 0, sfi.params(4, 16, 8, 0.3), 4)
    assert sfi.lib.sfi_ctx_create(ctypes.byref(desc), ctypes.byref(h)) == sfi.SFI_ERR_INVALID_ARG  # 0 layers
    desc = sfi.sfi_ctx_desc(2, 8, 2, 64, sfi.SFI_F32, 100, 1, sfi.params(4, 16, 8, 0.3), -1)
    assert sfi.lib.sfi_ctx_create(ctypes.byref(desc), ctypes.byref(h)) == sfi.SFI_ERR_INVALID_ARG  # budget < 0
    # refinements are checked like sfi_select_refined's
    for ref, code in [(sfi.sfi_refine(9, 0.5, 0.0), sfi.SFI_ERR_CAPACITY),
                      (sfi.sfi_refine(1, 0.0, 0.0), sfi.SFI_ERR_INVALID_ARG),
                      (sfi.sfi_refine(0, 1.0, -1.0), sfi.SFI_ERR_INVALID_ARG)]:
        desc = sfi.sfi_ctx_desc(2, 8, 2, 64, sfi.SFI_F32, 100, 1, sfi.params(4, 16, 8, 0.3), 4, 0, ref)
        assert sfi.lib.sfi_ctx_create(ctypes.byref(desc), ctypes.byref(h)) == code
    desc = sfi.sfi_ctx_desc(8, 32, 8, 128, sfi.SFI_BF16, 131072, 1, sfi.params(4, 256, 4096, 0.3), 32, 1,
                            sfi.sfi_refine(8, 0.5, 0.0))
    assert sfi.lib.sfi_ctx_create(ctypes.byref(desc), ctypes.byref(h)) == sfi.SFI_ERR_CAPACITY  # 131072 candidates
    assert sfi.lib.sfi_decode_step(None, 0, None, None, FAKE, FAKE, FAKE, FAKE, None) == sfi.SFI_ERR_INVALID_ARG


def test_schedule_matches_oracle(sfi):
    for budget in [0, 1, 3, 32]:
        tr = W.cfg2(n_steps=200).boundary_trace()
        ref = O.schedule(tr, budget)
        B = tr.shape[1]
        have = np.zeros(B, np.uint8)
        since = np.zeros(B, np.int32)
        for t in range(tr.shape[0]):
            got = sfi.sfi_schedule(tr[t], have, since, budget)
            assert list(got) == list(ref[t].astype(np.uint8)), (budget, t)
    with pytest.raises(sfi.SfiError):
        sfi.sfi_schedule(np.zeros(2, np.uint8), np.zeros(2, np.uint8), np.zeros(2, np.int32), -1)


def test_verify_validation_codes(sfi):
    """Verification attention rejects unsupported shapes and bad collected-row
    lists on the host (G = 4 here: n_rows * G may reach 32, every row may be
    collected)."""
    def verify(L, n_rows, collect, lsum=FAKE, ws=FAKE, q=FAKE):
        arr = (ctypes.c_int32 * max(1, len(collect)))(*collect) if collect is not None else None
        n = len(collect) if collect is not None else 0
        return sfi.lib.sfi_verify_attn(ctypes.byref(L), n_rows, arr, n, q, FAKE, FAKE, FAKE, lsum, ws,
                                       1 << 40, None)
    Lb = layout(sfi, dtype=sfi.SFI_BF16)
    assert verify(layout(sfi), 5, [0, 4]) == sfi.SFI_ERR_UNSUPPORTED           # fp32 cache
    assert verify(Lb, 0, [0]) == sfi.SFI_ERR_UNSUPPORTED
    assert verify(Lb, 9, [0]) == sfi.SFI_ERR_UNSUPPORTED                       # > 8 rows
    assert verify(layout(sfi, dtype=sfi.SFI_BF16, n_q_heads=16), 5, [0]) == sfi.SFI_ERR_UNSUPPORTED  # 5 * 8 > 32
    assert verify(Lb, 5, [0, 0]) == sfi.SFI_ERR_INVALID_ARG                    # repeated row
    assert verify(Lb, 5, [5]) == sfi.SFI_ERR_INVALID_ARG                       # row outside the chain
    assert verify(Lb, 5, [0, 1, 2, 3, 4, 0]) == sfi.SFI_ERR_INVALID_ARG        # more rows than the chain
    assert verify(Lb, 5, [0, 1, 2, 3, 4], q=None) == sfi.SFI_ERR_INVALID_ARG
    # every row collected passes the row checks and stops at the missing workspace
    assert verify(Lb, 5, [0, 1, 2, 3, 4], ws=None) == sfi.SFI_ERR_WORKSPACE
    assert verify(Lb, 8, list(range(8)), ws=None) == sfi.SFI_ERR_WORKSPACE


def test_refine_validation_codes(sfi):
    """Soft-NMS / exclusivity refinement: parameter limits and the candidate
    capacity are checked on the host."""
    L = layout(sfi)
    Lbig = layout(sfi, max_len=131072)

    def ref(p, r, lay=L, f=FAKE, ws=FAKE, ws_bytes=1 << 40):
        rp = ctypes.byref(r) if r is not None else None
        return sfi.lib.sfi_select_refined(ctypes.byref(lay), ctypes.byref(p), rp, f, FAKE, FAKE, FAKE,
                                          None, ws, ws_bytes, None)

    P = sfi.params(4, 16, 8, 0.3)
    R = sfi.sfi_refine
    assert ref(P, None) == sfi.SFI_ERR_INVALID_ARG
    assert ref(sfi.params(0, 5, 8, 0.0, mode=sfi.SFI_SELECT_LOGIT_SUM_HEAD), R(1, 0.5, 0.0)) == sfi.SFI_ERR_INVALID_ARG
    assert ref(P, R(-1, 0.5, 0.0)) == sfi.SFI_ERR_INVALID_ARG
    assert ref(P, R(9, 0.5, 0.0)) == sfi.SFI_ERR_CAPACITY
    for sig in (0.0, -1.0, float("nan"), float("inf")):
        assert ref(P, R(1, sig, 0.0)) == sfi.SFI_ERR_INVALID_ARG
    for beta in (-0.5, float("nan"), float("inf")):
        assert ref(P, R(0, 1.0, beta)) == sfi.SFI_ERR_INVALID_ARG
    # min(max_len, (k - 1)(4 rho + 1) + 1) candidates must fit the cluster's shared memory (98304)
    assert ref(sfi.params(4, 256, 4096, 0.3), R(8, 0.5, 0.0), lay=Lbig) == sfi.SFI_ERR_CAPACITY
    assert ref(sfi.params(4, 256, 4096, 0.3), R(2, 0.5, 0.0), lay=Lbig, ws=None) == sfi.SFI_ERR_WORKSPACE
    assert ref(P, R(1, 0.5, 0.2), f=None) == sfi.SFI_ERR_INVALID_ARG
    assert ref(P, R(1, 0.5, 0.2), ws_bytes=16) == sfi.SFI_ERR_WORKSPACE

    def size(p, r, lay=L):
        return sfi.lib.sfi_select_refined_workspace_size(ctypes.byref(lay), ctypes.byref(p), ctypes.byref(r))
    assert size(P, R(9, 0.5, 0.0)) == 0
    base = sfi.lib.sfi_select_workspace_size(ctypes.byref(L), ctypes.byref(P))
    # rho = 1: (8 - 1) * 5 + 1 = 36 candidates per unit, beside the counts and the plain plan
    assert size(P, R(1, 0.5, 0.0)) > size(P, R(0, 0.5, 0.0)) > base


def test_header_compiles_as_c99(tmp_path):
    """include/sfi.h is a C header: plain C99 (pedantic) compiles it, types and all."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "hdr.c"
    src.write_text('#include "sfi.h"\n'
                   "int main(void) {\n"
                   "  sfi_refine r = {1, 0.5f, 0.0f};\n"
                   "  sfi_ctx_desc d = {0};\n"
                   "  sfi_params p = {4, 256, 4096, 0.3f, SFI_SELECT_FUSED};\n"
                   "  d.params = p;\n"
                   "  d.refine = r;\n"
                   "  return (int)(sizeof d == 0) + (int)sfi_select_refined_workspace_size(0, &p, &r);\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        f"-I{os.path.join(ROOT, 'include')}", "-c", str(src), "-o", str(tmp_path / "hdr.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_wait_limit_setter(sfi):
    assert sfi.lib.sfi_set_wait_limit(-1) == sfi.SFI_ERR_INVALID_ARG
    assert "wait limit" in sfi.lib.sfi_last_error().decode()
    assert sfi.lib.sfi_set_wait_limit(12345) == sfi.SFI_OK
    assert sfi.lib.sfi_set_wait_limit(0) == sfi.SFI_OK  # back to the default
