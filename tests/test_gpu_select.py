"""The step after a verify with the rollback folded in (gdn_decode_step_select).

Reading each sequence's entering state from the snapshot its accepted count
selects must give exactly what committing (copying that snapshot back) and
then stepping gives: outputs, state and conv window, bit for bit, for the
K = 2 snapshot layout of gdn_verify_k2 and the generic one of gdn_verify_kn.
"""
import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import device_inputs, dims_of, params_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402


def _verify(form, K, dev, shape, prm):
    """K draft tokens (rows 0..K-1 of every sequence) through the verify call of `form`."""
    B, Hv, d, cd, W = shape.B, shape.Hv, shape.d, shape.conv_dim, shape.W
    toks = {k: dev[k][:, :K].contiguous() for k in ("x", "z", "alpha", "beta_logit")}
    vshape = synth.Shape(B=B, T=K, Hq=shape.Hq, Hv=Hv, warm=True)
    out = torch.empty(B, K, Hv, d, device="cuda")
    if form == "k2":
        ssnap = torch.empty(B, Hv, d, d, device="cuda")
        csnap = torch.empty(B, cd, W - 1, device="cuda")
        gdn.verify_k2(dev["state"], dev["hist"], ssnap, csnap, toks["x"], toks["z"], toks["alpha"],
                      toks["beta_logit"], prm, out, dims_of(vshape))
        entries = K - 1
    else:
        ssnap = torch.empty(B, K - 1, Hv, d, d, device="cuda")
        csnap = torch.empty(B, K, cd, W - 1, device="cuda")
        gdn.verify_kn(dev["state"], dev["hist"], ssnap, csnap, toks["x"], toks["z"], toks["alpha"],
                      toks["beta_logit"], prm, out, dims_of(vshape), K)
        entries = K
    return ssnap, csnap, entries


@pytest.mark.parametrize("form, K", [("k2", 2), ("kn", 2), ("kn", 4)])
def test_select_step_equals_commit_then_step(form, K):
    shape = synth.Shape(B=6, T=K + 1, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=80 + K)
    dev = device_inputs(shape, inp)
    prm = params_of(dev)
    B, Hv, d = shape.B, shape.Hv, shape.d
    ssnap, csnap, entries = _verify(form, K, dev, shape, prm)
    # a mix of accepted counts, the full draft and a single token among them
    acc = torch.tensor([(b % K) + 1 for b in range(B)], dtype=torch.int32, device="cuda")
    assert set(acc.tolist()) == set(range(1, K + 1))
    step_dims = dims_of(shape, rows_per_seq=K + 1)
    tok = {k: dev[k][:, K] for k in ("x", "z", "alpha", "beta_logit")}
    # commit, then the next token
    st_a, hi_a = dev["state"].clone(), dev["hist"].clone()
    if form == "k2":
        gdn.verify_commit(st_a, hi_a, ssnap, csnap, acc, dims_of(shape))
    else:
        gdn.verify_commit_kn(st_a, hi_a, ssnap, csnap, acc, dims_of(shape), K)
    out_a = torch.empty(B, Hv, d, device="cuda")
    gdn.decode_step(st_a, hi_a, tok["x"], tok["z"], tok["alpha"], tok["beta_logit"], prm, out_a,
                    step_dims)
    # the next token straight from the selected snapshots
    st_b, hi_b = dev["state"].clone(), dev["hist"].clone()
    out_b = torch.empty(B, Hv, d, device="cuda")
    gdn.decode_step_select(st_b, hi_b, ssnap, csnap, entries, acc, K, tok["x"], tok["z"],
                           tok["alpha"], tok["beta_logit"], prm, out_b, step_dims)
    torch.cuda.synchronize()
    assert gdn.check_device() == 0
    assert torch.equal(out_a, out_b)
    assert torch.equal(st_a, st_b)
    assert torch.equal(hi_a, hi_b)


def test_select_step_flags_out_of_range_counts():
    K = 3
    shape = synth.Shape(B=4, T=K + 1, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=90)
    dev = device_inputs(shape, inp)
    prm = params_of(dev)
    B, Hv, d = shape.B, shape.Hv, shape.d
    ssnap, csnap, entries = _verify("kn", K, dev, shape, prm)
    step_dims = dims_of(shape, rows_per_seq=K + 1)
    tok = {k: dev[k][:, K] for k in ("x", "z", "alpha", "beta_logit")}
    assert gdn.check_device() == 0
    # 0 and K + 1 are out of range: those sequences start from the live state, like K
    acc = torch.tensor([0, K, K + 1, -5], dtype=torch.int32, device="cuda")
    st_b, hi_b = dev["state"].clone(), dev["hist"].clone()
    out_b = torch.empty(B, Hv, d, device="cuda")
    gdn.decode_step_select(st_b, hi_b, ssnap, csnap, entries, acc, K, tok["x"], tok["z"],
                           tok["alpha"], tok["beta_logit"], prm, out_b, step_dims)
    assert gdn.check_device() == 16
    st_a, hi_a = dev["state"].clone(), dev["hist"].clone()
    out_a = torch.empty(B, Hv, d, device="cuda")
    gdn.decode_step(st_a, hi_a, tok["x"], tok["z"], tok["alpha"], tok["beta_logit"], prm, out_a,
                    step_dims)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(st_a, st_b) and torch.equal(hi_a, hi_b)
    assert gdn.check_device() == 0
