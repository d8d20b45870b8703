"""Bounded waits on the GPU: a kernel whose wait runs out reports it and returns.

The first wait of the chunked prefill's sequential pass and each CTA's first
tile-copy wait in the multi-token conv take their limit from a test hook
(include/gdn_testing.h). Set to 1 ns, those waits give up while the work they
wait for is still in flight: the kernels must set their bit of the device
error word, drain the copies they issued, free their tensor memory and return,
and the next call with the default limit must give correct results. Nothing
here faults or hangs the GPU: the waits end by their own limits.
"""
import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import (STATE_TOL, check_out, device_inputs, dims_of, max_rel, params_of,
                         run_oracle)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402

BIT_PREFILL_CHAIN = 1
BIT_CONV_TILE = 64


def _prefill(shape, dev):
    out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
    gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                        dev["beta_logit"], params_of(dev), out, dims_of(shape), shape.T, 64)
    return out


def test_prefill_wait_expiry_is_reported_and_the_next_call_is_correct():
    shape = synth.Shape(B=2, T=150, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=61)
    assert gdn.check_device() == 0
    gdn.testing_set_first_wait_ns(1)
    try:
        dev = device_inputs(shape, inp)
        _prefill(shape, dev)
        code = gdn.check_device()
    finally:
        gdn.testing_set_first_wait_ns(0)
    assert code & BIT_PREFILL_CHAIN, code
    assert not code & 8, code            # every issued copy drained
    # the context is intact: a fresh call with the default limit is correct
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    out = _prefill(shape, dev)
    torch.cuda.synchronize()
    assert gdn.check_device() == 0
    check_out(out.cpu().numpy(), ref["out"], y=ref["y"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL


def test_tiled_conv_wait_expiry_is_reported_and_the_next_call_is_correct():
    shape = synth.Shape(B=2, T=200, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=62)
    dims = dims_of(shape)
    assert gdn.check_device() == 0
    gdn.testing_set_first_wait_ns(1)
    try:
        dev = device_inputs(shape, inp)
        out = torch.empty(shape.B, shape.T, shape.conv_dim, device="cuda")
        gdn.conv_update(dev["hist"], dev["x"], dev["conv_w"], out, dims, shape.T)
        code = gdn.check_device()
    finally:
        gdn.testing_set_first_wait_ns(0)
    assert code & BIT_CONV_TILE, code
    # the multi-token conv with the default limit equals single-token calls bit for bit
    dev = device_inputs(shape, inp)
    out = torch.empty(shape.B, shape.T, shape.conv_dim, device="cuda")
    h0 = dev["hist"].clone()
    gdn.conv_update(dev["hist"], dev["x"], dev["conv_w"], out, dims, shape.T)
    step = torch.empty(shape.B, 1, shape.conv_dim, device="cuda")
    ref = torch.empty_like(out)
    d1 = dims_of(shape, rows_per_seq=shape.T)
    for t in range(shape.T):
        gdn.conv_update(h0, dev["x"][:, t], dev["conv_w"], step, d1, 1)
        ref[:, t] = step[:, 0]
    torch.cuda.synchronize()
    assert gdn.check_device() == 0
    assert torch.equal(out, ref)
    assert torch.equal(dev["hist"], h0)
