"""GPU parity on the method's degenerate inputs, against the fp64 oracle.

Each case sets some gates or activations to the values where the arithmetic
takes a special path:
  full forget  A_log = 10: the decay exp(g) underflows to exactly 0, so the
               state is rebuilt from the current token alone;
  no decay     alpha = -100: softplus ~ e^-100, g ~ 0, decay 1;
  guard        alpha + dt exactly 20 (log1p(exp(20)) branch), 20.5 and 30
               (identity branch) and 19.5 ("fm_kernel_ssm.h", "Decay gate":
               the softplus is the identity strictly above 20);
  beta zero    beta_logit = -100: sigmoid rounds to 0 on the GPU (e^100
               overflows float32), to 3.7e-44 in the oracle: no update;
  zero Q/K     Q/K inputs and history zero: the L2 norm returns
               0 / sqrt(eps) = 0, so k = q = 0 (no update, zero readout) and the
               state only decays (mildly: A_log = -2).
Every case runs through single-token decode steps, the chunked prefill and
the fused layer scan.
"""
import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import (check_out, OUT_TOL, STATE_TOL, device_inputs, dims_of, max_rel, out_rel, params_of,
                         run_oracle)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402


def _bf16(v):
    return synth.bf16_round(np.asarray(v, np.float32))


def _case(name, T):
    shape = synth.Shape(B=2, T=T, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=80 + T)
    Hv, d, Hq = shape.Hv, shape.d, shape.Hq
    if name == "full_forget":
        inp["A_log"][: Hv // 2] = 10.0
    elif name == "no_decay":
        inp["alpha"][:, ::2, :] = _bf16(-100.0)
    elif name == "guard":
        inp["dt"][:] = 0.5
        vals = _bf16([19.5, 20.0, 29.5, 19.0])      # alpha + dt = 20, 20.5, 30, 19.5
        inp["alpha"][...] = vals[np.arange(T)[:, None] % 4][None, :, :].repeat(Hv, -1)[..., :Hv]
    elif name == "beta_zero":
        inp["beta_logit"][:, 1::2, :] = _bf16(-100.0)
    elif name == "zero_qk":
        inp["x"][:, :, : 2 * Hq * d] = _bf16(0.0)   # all Q/K inputs of every token
        inp["hist"][:, : 2 * Hq * d, :] = 0.0
        # with no update the state only decays; keep the decay mild so that after 70
        # tokens it is still far above float32's range limit (a decay to exactly zero
        # is the full-forget case)
        inp["A_log"][:] = -2.0
    else:
        raise ValueError(name)
    return shape, inp


CASES = ["full_forget", "no_decay", "guard", "beta_zero", "zero_qk"]


@pytest.mark.parametrize("name", CASES)
def test_degenerate_decode_steps(name):
    shape, inp = _case(name, T=5)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    dims = dims_of(shape, rows_per_seq=shape.T)
    out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
    one = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    for t in range(shape.T):
        gdn.decode_step(dev["state"], dev["hist"], dev["x"][:, t], dev["z"][:, t],
                        dev["alpha"][:, t], dev["beta_logit"][:, t], params_of(dev), one, dims)
        out[:, t] = one
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.isfinite(o).all()
    check_out(o, ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    if name == "zero_qk":
        assert not o.any()


@pytest.mark.parametrize("name", CASES)
def test_degenerate_prefill_and_layer_scan(name):
    shape, inp = _case(name, T=70)
    ref = run_oracle(shape, inp, readout=True)
    for fn in ("prefill", "scan"):
        dev = device_inputs(shape, inp)
        out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
        if fn == "prefill":
            gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                                dev["beta_logit"], params_of(dev), out, dims_of(shape), shape.T, 64)
        else:
            gdn.layer_scan(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                           dev["beta_logit"], params_of(dev), out, dims_of(shape), shape.T)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        assert np.isfinite(o).all(), fn
        check_out(o, ref["out"], what=fn, y=ref["y"])
        assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL, fn
        assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32)), fn
