"""GPU parity of the chunked prefill against the fp64 sequential-scan oracle."""
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

PREFILL_STATE_TOL = STATE_TOL


def _prefill(shape, dev, T=None):
    T = shape.T if T is None else T
    out = torch.empty(shape.B, T, shape.Hv, shape.d, device="cuda")
    gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                        dev["beta_logit"], params_of(dev), out, dims_of(shape), T, 64)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 200])
@pytest.mark.parametrize("warm", [False, True])
def test_prefill_ragged_lengths_match_oracle(T, warm):
    shape = synth.Shape(B=2, T=T, Hq=2, Hv=4, warm=warm)
    inp = synth.make_inputs(shape, seed=300 + T)
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    out = _prefill(shape, dev).cpu().numpy()
    check_out(out, ref["out"], y=ref["y"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


@pytest.mark.parametrize("W,Hq,Hv", [(2, 1, 3), (8, 2, 2), (4, 1, 8)])
def test_prefill_edge_shapes(W, Hq, Hv):
    shape = synth.Shape(B=1, T=150, Hq=Hq, Hv=Hv, W=W, warm=True)
    inp = synth.make_inputs(shape, seed=400 + W)
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    out = _prefill(shape, dev).cpu().numpy()
    check_out(out, ref["out"], y=ref["y"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


def test_prefill_fp32_activations():
    shape = synth.Shape(B=1, T=130, Hq=4, Hv=4, act_dtype="f32", warm=True)
    inp = synth.make_inputs(shape, seed=31)
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    out = _prefill(shape, dev).cpu().numpy()
    check_out(out, ref["out"], y=ref["y"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL


def test_prefill_with_unaligned_z_rows():
    # z rows an odd number of bf16 elements apart cannot be staged by 16-byte copies;
    # the kernel reads them directly instead
    shape = synth.Shape(B=2, T=130, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=35)
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    zs = shape.Hv * shape.d + 1
    zpad = torch.zeros(shape.B, shape.T, zs, dtype=dev["z"].dtype, device="cuda")
    zpad[..., :shape.Hv * shape.d] = dev["z"]
    dims = dims_of(shape)
    dims.z_stride = zs
    out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
    gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], zpad, dev["alpha"], dev["beta_logit"],
                        params_of(dev), out, dims, shape.T, 64)
    torch.cuda.synchronize()
    check_out(out.cpu().numpy(), ref["out"], y=ref["y"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL


def test_prefill_then_decode_continues_the_sequence():
    # prefill T tokens then decode one more == oracle over T + 1 tokens
    shape = synth.Shape(B=2, T=97, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=32)
    ref = run_oracle(shape, inp, readout=True)
    dev = device_inputs(shape, inp)
    T = shape.T - 1
    xs = {k: dev[k][:, :T].contiguous() for k in ("x", "z", "alpha", "beta_logit")}
    out = torch.empty(shape.B, T, shape.Hv, shape.d, device="cuda")
    gdn.prefill_chunked(dev["state"], dev["hist"], xs["x"], xs["z"], xs["alpha"], xs["beta_logit"],
                        params_of(dev), out, dims_of(shape), T, 64)
    step = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    last = {k: dev[k][:, T].contiguous() for k in ("x", "z", "alpha", "beta_logit")}
    gdn.decode_step(dev["state"], dev["hist"], last["x"], last["z"], last["alpha"],
                    last["beta_logit"], params_of(dev), step, dims_of(shape))
    torch.cuda.synchronize()
    check_out(out.cpu().numpy(), ref["out"][:, :T], y=ref["y"][:, :T])
    check_out(step.cpu().numpy(), ref["out"][:, T], y=ref["y"][:, T])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


def test_prefill_full_size_4x8192():
    # the full prefill workload; the oracle scans every token for the final state and
    # its outputs are compared on each sequence's first 512 tokens and last chunk
    shape = synth.WORKLOADS["prefill"]
    inp = synth.make_inputs(shape, seed=4)
    dev = device_inputs(shape, inp)
    out = _prefill(shape, dev)
    ref = run_oracle(shape, inp, readout=True)
    o = out.cpu().numpy()
    check_out(o[:, :512], ref["out"][:, :512], y=ref["y"][:, :512])
    check_out(o[:, -64:], ref["out"][:, -64:], y=ref["y"][:, -64:])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


def test_prefill_explicit_workspace_contents_do_not_matter():
    # a caller-owned workspace filled with garbage and reused by two calls in a row
    shape = synth.Shape(B=2, T=200, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=36)
    ref = run_oracle(shape, inp, readout=True)
    dims = dims_of(shape)
    nbytes = gdn.prefill_workspace_bytes(dims, shape.T)
    assert nbytes == shape.B * 4 * (shape.Hv * 34816 + shape.Hq * 65536)
    ws = torch.full((nbytes + 4096,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN bit patterns
    outs = []
    for _ in range(2):
        dev = device_inputs(shape, inp)
        out = torch.empty(shape.B, shape.T, shape.Hv, shape.d, device="cuda")
        gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                            dev["beta_logit"], params_of(dev), out, dims, shape.T, 64, workspace=ws)
        torch.cuda.synchronize()
        check_out(out.cpu().numpy(), ref["out"], y=ref["y"])
        assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= PREFILL_STATE_TOL
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    with pytest.raises(gdn.GdnError):
        gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                            dev["beta_logit"], params_of(dev), out, dims, shape.T, 64,
                            workspace=ws[:nbytes - 16])
