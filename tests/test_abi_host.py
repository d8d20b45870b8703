"""C-ABI checks that need no GPU: the library loads, exports every function
include/gdn.h declares, and rejects bad arguments on the host before any
CUDA call is made."""
import ctypes as ct
import os
import re

import pytest

import gated_delta_ssm_gb300 as gdn
from gated_delta_ssm_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gdn_conv_update", "gdn_decay_gate", "gdn_recurrence_decode", "gdn_verify_k2",
                     "gdn_prefill_chunked", "gdn_gated_norm", "gdn_decode_step",
                     "gdn_verify_commit", "gdn_recurrence_scan", "gdn_layer_scan",
                     "gdn_verify_kn", "gdn_verify_commit_kn", "gdn_last_cuda_error",
                     "gdn_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.gdn_version()
    assert lib.gdn_status_string(1) == b"GDN_ERR_INVALID_ARG"
    assert lib.gdn_last_cuda_error() == b""


FAKE = 1 << 40      # a well-aligned non-null address; never dereferenced on these paths


def _dims(**kw):
    d = dict(n_seq=2, n_qk_heads=2, n_v_heads=4, head_dim=128, d_conv=4)
    d.update(kw)
    return gdn.Dims(**d)


def _params():
    return gdn.Params(FAKE, FAKE, FAKE, FAKE)


def _decode(lib, dims, **ptrs):
    p = dict(state=FAKE, conv=FAKE, x=FAKE, z=FAKE, a=FAKE, b=FAKE, out=FAKE)
    p.update(ptrs)
    cd, cp = dims.c(), _params().c()
    return lib.gdn_decode_step(p["state"], p["conv"], p["x"], p["z"], p["a"], p["b"], gdn.GDN_BF16,
                               ct.byref(cp), p["out"], ct.byref(cd), None)


@pytest.mark.parametrize("field", ["state", "conv", "x", "z", "a", "b", "out"])
def test_decode_step_rejects_null_pointers(lib, field):
    assert _decode(lib, _dims(), **{field: None}) == gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    (dict(n_seq=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(n_seq=65536), gdn.GDN_ERR_INVALID_ARG),                    # one past the grid limit
    (dict(n_qk_heads=3, n_v_heads=4), gdn.GDN_ERR_INVALID_ARG),      # Hv not a multiple of Hq
    (dict(head_dim=64), gdn.GDN_ERR_UNSUPPORTED),
    (dict(d_conv=1), gdn.GDN_ERR_UNSUPPORTED),
    (dict(d_conv=9), gdn.GDN_ERR_UNSUPPORTED),
    (dict(n_qk_heads=1, n_v_heads=16), gdn.GDN_ERR_UNSUPPORTED),     # r = 16 > 8
    (dict(x_stride=100), gdn.GDN_ERR_INVALID_ARG),
    (dict(z_stride=5), gdn.GDN_ERR_INVALID_ARG),
    (dict(gate_stride=3), gdn.GDN_ERR_INVALID_ARG),
])
def test_decode_step_rejects_bad_dims(lib, kw, status):
    assert _decode(lib, _dims(**kw)) == status


def test_decode_step_rejects_misaligned_state(lib):
    assert _decode(lib, _dims(), state=FAKE + 4) == gdn.GDN_ERR_INVALID_ARG
    assert _decode(lib, _dims(), x=FAKE + 1) == gdn.GDN_ERR_INVALID_ARG


def test_verify_rejects_aliased_snapshot(lib):
    cd, cp = _dims().c(), _params().c()
    st = lib.gdn_verify_k2(FAKE, FAKE + 64, FAKE, FAKE + 128, FAKE, FAKE, FAKE, FAKE, gdn.GDN_F32,
                           ct.byref(cp), FAKE, ct.byref(cd), None)
    assert st == gdn.GDN_ERR_INVALID_ARG


def test_prefill_rejects_bad_chunk_and_tokens(lib):
    cd, cp = _dims().c(), _params().c()
    args = [FAKE] * 6 + [gdn.GDN_BF16, ct.byref(cp), FAKE, ct.byref(cd)]
    ws = 1 << 30
    assert lib.gdn_prefill_chunked(*args, 128, 32, FAKE, ws, None) == gdn.GDN_ERR_UNSUPPORTED
    assert lib.gdn_prefill_chunked(*args, 0, 64, FAKE, ws, None) == gdn.GDN_ERR_INVALID_ARG


def test_prefill_workspace_size_and_checks(lib):
    # per (sequence, 64-token chunk): a 34 KB image per V head and a 64 KB image per QK head
    dims = _dims()
    cd, cp = dims.c(), _params().c()
    for T, chunks in ((1, 1), (64, 1), (65, 2), (8192, 128)):
        assert gdn.prefill_workspace_bytes(dims, T) == 2 * chunks * (4 * 34816 + 2 * 65536)
    assert gdn.prefill_workspace_bytes(dims, 0) == 0
    assert gdn.prefill_workspace_bytes(dims, 64, 32) == 0
    need = gdn.prefill_workspace_bytes(dims, 130)
    args = [FAKE] * 6 + [gdn.GDN_BF16, ct.byref(cp), FAKE, ct.byref(cd), 130, 64]
    # missing, too small, or misaligned workspace
    assert lib.gdn_prefill_chunked(*args, None, need, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_prefill_chunked(*args, FAKE, need - 1, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_prefill_chunked(*args, FAKE + 8, need, None) == gdn.GDN_ERR_INVALID_ARG


def test_testing_header_hook_is_exported(lib):
    text = open(os.path.join(ROOT, "include", "gdn_testing.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for name in set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)):
        assert hasattr(lib, name), name


def test_row_splits_follow_the_sm_count(lib):
    # the launchers size their grids from the device's SM count, not a fixed 152
    for sms in (20, 132, 148, 152, 160, 170):
        for B in (1, 2, 4, 32, 64):
            for Hv in (8, 32, 48):
                for r in (1, 2, 4):
                    dec, scan = gdn.testing_row_splits(B, Hv, r, sms)
                    assert dec in (1, 2, 4) and scan in (1, 2, 4)
                    assert r * dec <= 8 and r * scan <= 8        # one cluster of r x split CTAs
                    # the scans never spill a partial second wave of 2 CTAs per SM by splitting
                    assert scan == 1 or B * Hv * scan <= 2 * sms
                    # and split as far as that allows
                    if scan < 4 and r * scan * 2 <= 8:
                        assert B * Hv * scan * 2 > 2 * sms
                    # the decode splits until about four CTAs per SM, or until a further
                    # split would grow a cluster past 4 CTAs
                    assert dec == 1 or r * dec <= 4
                    if dec < 4 and r * dec * 2 <= 4:
                        assert B * Hv * dec >= 4 * sms
    # the GB300's 152 SMs: the benchmarked shapes keep their splits
    assert gdn.testing_row_splits(1, 32, 2, 152) == (2, 4)     # one sequence, 16 / 32 heads
    assert gdn.testing_row_splits(64, 48, 3, 152) == (1, 1)    # 64 sequences, 16 / 48 heads
    assert gdn.testing_row_splits(32, 32, 2, 152) == (1, 1)    # 32 sequences, 16 / 32 heads


def test_other_entry_points_validate(lib):
    cd = _dims().c()
    assert lib.gdn_decay_gate(None, 0, 4, FAKE, FAKE, FAKE, 1, 4, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_decay_gate(FAKE, 0, 3, FAKE, FAKE, FAKE, 1, 4, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_conv_update(FAKE, FAKE, 0, FAKE, FAKE, ct.byref(cd), 0, 1e-6, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_gated_norm(FAKE, FAKE, FAKE, 0, 512, FAKE, 1, 4, 64, 1e-6, None) == gdn.GDN_ERR_UNSUPPORTED
    assert lib.gdn_gated_norm(FAKE, FAKE, FAKE, 0, 100, FAKE, 1, 4, 128, 1e-6, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_recurrence_decode(FAKE, FAKE, FAKE, FAKE, 10, FAKE, FAKE, FAKE, ct.byref(cd),
                                     1.0, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_commit(FAKE, FAKE, FAKE, FAKE, None, ct.byref(cd), None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 7, ct.byref(_params().c()), FAKE,
                               ct.byref(cd), None) == gdn.GDN_ERR_INVALID_ARG


def test_scan_entry_points_validate(lib):
    cd, cp = _dims().c(), _params().c()
    # recurrence scan: n_tokens < 1, qkv_stride too small, null y
    rs = lambda stride, n, y=FAKE: lib.gdn_recurrence_scan(FAKE, FAKE, FAKE, FAKE, stride, FAKE,
                                                           FAKE, y, ct.byref(cd), n, 1.0, None)
    assert rs(1536, 0) == gdn.GDN_ERR_INVALID_ARG
    assert rs(10, 4) == gdn.GDN_ERR_INVALID_ARG
    assert rs(1536, 4, None) == gdn.GDN_ERR_INVALID_ARG
    layer = [FAKE] * 6 + [gdn.GDN_BF16, ct.byref(cp), FAKE, ct.byref(cd)]
    assert lib.gdn_layer_scan(*layer, 0, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_layer_scan(*([FAKE + 4] + layer[1:]), 3, None) == gdn.GDN_ERR_INVALID_ARG
    bad_w = gdn.Dims(n_seq=2, n_qk_heads=2, n_v_heads=4, d_conv=9).c()
    assert lib.gdn_layer_scan(*layer[:9], ct.byref(bad_w), 3, None) == gdn.GDN_ERR_UNSUPPORTED


def test_select_step_validates(lib):
    # every case below fails on the host before a launch (the pointers are never dereferenced)
    cd, cp = _dims().c(), _params().c()
    tail = [FAKE] * 4 + [gdn.GDN_F32, ct.byref(cp), FAKE, ct.byref(cd), None]
    G = 1 << 30                      # far apart: no overlap between these ranges
    st, conv, ss, cs, acc = FAKE, FAKE + G, FAKE + 2 * G, FAKE + 3 * G, FAKE + 4 * G
    sel = lambda *a: lib.gdn_decode_step_select(*a, *tail)
    assert sel(st, conv, ss, cs, 2, None, 2) == gdn.GDN_ERR_INVALID_ARG        # no counts
    assert sel(st, conv, ss, cs, 2, acc, 0) == gdn.GDN_ERR_INVALID_ARG         # n_draft < 1
    assert sel(st, conv, None, cs, 2, acc, 3) == gdn.GDN_ERR_INVALID_ARG       # no state snapshots
    assert sel(st, conv, ss, None, 3, acc, 3) == gdn.GDN_ERR_INVALID_ARG       # no conv snapshots
    assert sel(st, conv, ss, cs, 1, acc, 3) == gdn.GDN_ERR_INVALID_ARG         # entries not K-1 or K
    assert sel(st, conv, ss, cs, 4, acc, 3) == gdn.GDN_ERR_INVALID_ARG
    assert sel(st, conv, st + 64, cs, 3, acc, 3) == gdn.GDN_ERR_INVALID_ARG    # snapshot inside state
    assert sel(st, conv, ss, conv + 64, 3, acc, 3) == gdn.GDN_ERR_INVALID_ARG  # inside conv_state


def test_verify_kn_requires_distinct_snapshots(lib):
    cd, cp = _dims().c(), _params().c()
    tail = [FAKE] * 4 + [gdn.GDN_F32, ct.byref(cp), FAKE, ct.byref(cd)]
    st, conv, ss, cs = FAKE, FAKE + 64, FAKE + 128, FAKE + 192
    assert lib.gdn_verify_kn(st, conv, None, cs, *tail, 3, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_kn(st, conv, ss, None, *tail, 3, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_kn(st, conv, st, cs, *tail, 3, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_kn(st, conv, ss, conv, *tail, 3, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_kn(st, conv, ss, cs, *tail, 0, None) == gdn.GDN_ERR_INVALID_ARG
    commit = lambda ss_, n: lib.gdn_verify_commit_kn(st, conv, ss_, cs, FAKE, ct.byref(cd), n, None)
    assert commit(ss, 0) == gdn.GDN_ERR_INVALID_ARG
    assert commit(None, 3) == gdn.GDN_ERR_INVALID_ARG
    assert commit(ss + 4, 3) == gdn.GDN_ERR_INVALID_ARG


def test_binding_raises_loudly_on_bad_status(lib):
    with pytest.raises(gdn.GdnError):
        gdn._check(gdn.GDN_ERR_INVALID_ARG, "gdn_decode_step")


def test_header_is_plain_c99(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "uses_header.c"
    src.write_text('#include "gdn.h"\nint main(void) { return (int)GDN_OK + (int)sizeof(gdn_dims); }\n')
    r = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_client_compiles_as_c():
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = "/usr/local/cuda/include"
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                        os.path.join(ROOT, "tests", "c_client", "gdn_c_client.c")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
