"""The allocation-free prefill entry point, through the C ABI.

gdn_prefill_chunked_noalloc serves callers that cannot allocate device memory
(a runtime whose device memory is all planned at start-up, or a loop that must
not pay for an allocation): its workspace is a fixed array inside the library.
It must give the same results as gdn_prefill_chunked with a caller-owned
workspace, call after call, since every call reuses the same array. This file
is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes as ct

import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import OUT_TOL, STATE_TOL, device_inputs, dims_of, max_rel, out_rel, params_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402

STATIC_SCRATCH = 16 << 20


def _noalloc_fn():
    lib = gdn.load()
    fn = lib.gdn_prefill_chunked_noalloc
    vp = ct.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ct.c_int, vp, vp, vp, ct.c_int32, ct.c_int32, vp]
    fn.restype = ct.c_int
    return fn


def _call_noalloc(fn, shape, dev, out, dims):
    cd, cp = dims.c(), params_of(dev).c()
    return fn(dev["state"].data_ptr(), dev["hist"].data_ptr(), dev["x"].data_ptr(),
              dev["z"].data_ptr(), dev["alpha"].data_ptr(), dev["beta_logit"].data_ptr(),
              gdn.GDN_BF16, ct.addressof(cp), out.data_ptr(), ct.addressof(cd), shape.T, 64,
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_prefill_matches_the_workspace_entry_point_twice_in_a_row():
    fn = _noalloc_fn()
    shape = synth.Shape(B=2, T=200, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=71)
    dims = dims_of(shape)
    # the existing entry point with a caller-owned workspace
    ref = device_inputs(shape, inp)
    ref_out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
    ws = torch.empty(gdn.prefill_workspace_bytes(dims, shape.T), dtype=torch.uint8, device="cuda")
    gdn.prefill_chunked(ref["state"], ref["hist"], ref["x"], ref["z"], ref["alpha"],
                        ref["beta_logit"], params_of(ref), ref_out, dims, shape.T, 64, workspace=ws)
    torch.cuda.synchronize()
    ro, rs, rh = ref_out.cpu().numpy(), ref["state"].cpu().numpy(), ref["hist"].cpu().numpy()
    for _ in range(2):
        dev = device_inputs(shape, inp)
        out = torch.empty_like(ref_out)
        st = _call_noalloc(fn, shape, dev, out, dims)
        torch.cuda.synchronize()
        assert st == gdn.GDN_OK, st
        assert gdn.check_device() == 0
        assert out_rel(out.cpu().numpy(), ro) <= OUT_TOL
        assert max_rel(dev["state"].cpu().numpy(), rs, 2) <= STATE_TOL
        assert np.array_equal(dev["hist"].cpu().numpy(), rh)


def test_noalloc_prefill_rejects_work_beyond_its_scratch():
    fn = _noalloc_fn()
    # 2 sequences x 129 chunks x (4 x 34 KB + 2 x 64 KB) = 68 MB > 16 MiB
    shape = synth.Shape(B=2, T=129 * 64, Hq=2, Hv=4, warm=True)
    dims = dims_of(shape)
    assert gdn.prefill_workspace_bytes(dims, shape.T) > STATIC_SCRATCH
    small = synth.Shape(B=2, T=1, Hq=2, Hv=4, warm=True)
    dev = device_inputs(small, synth.make_inputs(small, seed=72))
    out = torch.empty(1, device="cuda")
    st = _call_noalloc(fn, shape, dev, out, dims)
    assert st == gdn.GDN_ERR_UNSUPPORTED
    assert b"static scratch" in gdn.load().gdn_last_cuda_error()
