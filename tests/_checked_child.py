"""Run by tests/test_gpu_checked.py in a child process with GDN_CHECKED=1: every
kernel family of the checked library (index range checks compiled in) on the
smallest shapes (one sequence, one V head) and ragged token counts. Exits 0
when no check fired (device error word 0) and the results match the oracle."""
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import gated_delta_ssm_gb300 as gdn  # noqa: E402
from gated_delta_ssm_gb300 import synth  # noqa: E402
from tests._util import (STATE_TOL, check_out, device_inputs, dims_of,  # noqa: E402
                         max_rel, params_of, run_oracle)


def expect_clean(what):
    torch.cuda.synchronize()
    code = gdn.check_device()
    if code != 0:
        raise SystemExit(f"{what}: device error word {code}")


def main():
    assert os.path.basename(gdn.library_path()) == "libgdn_checked.so", gdn.library_path()
    assert gdn.check_device() == 0
    for T in (1, 37, 130):
        shape = synth.Shape(B=1, T=T, Hq=1, Hv=1, warm=True)
        inp = synth.make_inputs(shape, seed=500 + T)
        ref = run_oracle(shape, inp, readout=True)
        prm_dims = dims_of(shape)
        # chunked prefill (ragged last chunk)
        dev = device_inputs(shape, inp)
        out = torch.empty(1, T, 1, shape.d, device="cuda")
        gdn.prefill_chunked(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                            dev["beta_logit"], params_of(dev), out, prm_dims, T, 64)
        expect_clean(f"prefill T={T}")
        check_out(out.cpu().numpy(), ref["out"], y=ref["y"])
        assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
        # layer scan
        dev = device_inputs(shape, inp)
        out = torch.empty(1, T, 1, shape.d, device="cuda")
        gdn.layer_scan(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                       dev["beta_logit"], params_of(dev), out, prm_dims, T)
        expect_clean(f"layer scan T={T}")
        check_out(out.cpu().numpy(), ref["out"], y=ref["y"])
        assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
        # multi-token conv (tiled for bf16 rows) and the token-serial conv of one step
        dev = device_inputs(shape, inp)
        conv = torch.empty(1, T, shape.conv_dim, device="cuda")
        gdn.conv_update(dev["hist"], dev["x"], dev["conv_w"], conv, prm_dims, T)
        expect_clean(f"conv T={T}")
    # single-token paths and the verify family
    for K in (2, 3):
        shape = synth.Shape(B=1, T=K + 1, Hq=1, Hv=1, warm=True)
        inp = synth.make_inputs(shape, seed=600 + K)
        dev = device_inputs(shape, inp)
        prm = params_of(dev)
        d, cd, W = shape.d, shape.conv_dim, shape.W
        toks = {k: dev[k][:, :K].contiguous() for k in ("x", "z", "alpha", "beta_logit")}
        vdims = dims_of(synth.Shape(B=1, T=K, Hq=1, Hv=1, warm=True))
        vout = torch.empty(1, K, 1, d, device="cuda")
        if K == 2:
            ssnap = torch.empty(1, 1, d, d, device="cuda")
            csnap = torch.empty(1, cd, W - 1, device="cuda")
            gdn.verify_k2(dev["state"], dev["hist"], ssnap, csnap, toks["x"], toks["z"], toks["alpha"],
                          toks["beta_logit"], prm, vout, vdims)
            entries = 1
        else:
            ssnap = torch.empty(1, K - 1, 1, d, d, device="cuda")
            csnap = torch.empty(1, K, cd, W - 1, device="cuda")
            gdn.verify_kn(dev["state"], dev["hist"], ssnap, csnap, toks["x"], toks["z"], toks["alpha"],
                          toks["beta_logit"], prm, vout, vdims, K)
            entries = K
        expect_clean(f"verify K={K}")
        acc = torch.ones(1, dtype=torch.int32, device="cuda")
        step_dims = dims_of(shape, rows_per_seq=K + 1)
        one = torch.empty(1, 1, d, device="cuda")
        st, hi = dev["state"].clone(), dev["hist"].clone()
        gdn.decode_step_select(st, hi, ssnap, csnap, entries, acc, K, dev["x"][:, K], dev["z"][:, K],
                               dev["alpha"][:, K], dev["beta_logit"][:, K], prm, one, step_dims)
        expect_clean(f"select step K={K}")
        if K == 2:
            gdn.verify_commit(dev["state"], dev["hist"], ssnap, csnap, acc, dims_of(shape))
        else:
            gdn.verify_commit_kn(dev["state"], dev["hist"], ssnap, csnap, acc, dims_of(shape), K)
        gdn.decode_step(dev["state"], dev["hist"], dev["x"][:, K], dev["z"][:, K], dev["alpha"][:, K],
                        dev["beta_logit"][:, K], prm, one, step_dims)
        expect_clean(f"commit + step K={K}")
        assert torch.equal(st, dev["state"]) and torch.equal(hi, dev["hist"])
    # the standalone parts
    shape = synth.Shape(B=1, T=5, Hq=1, Hv=1, warm=True)
    inp = synth.make_inputs(shape, seed=700)
    ref = run_oracle(shape, inp, intermediates=True)
    dev = device_inputs(shape, inp)
    d, cd = shape.d, shape.conv_dim
    conv = torch.from_numpy(ref["conv"].astype(np.float32)).cuda()
    g = torch.from_numpy(ref["g"].astype(np.float32)).cuda()
    beta = torch.from_numpy(ref["beta"].astype(np.float32)).cuda()
    y = torch.empty(1, 5, 1, d, device="cuda")
    gdn.recurrence_scan(dev["state"].clone(), conv, conv[..., d:], conv[..., 2 * d:], cd, g, beta, y,
                        dims_of(shape), 5, 1 / math.sqrt(d))
    gdn.recurrence_decode(dev["state"].clone(), conv[:, 0], conv[:, 0, d:], conv[:, 0, 2 * d:],
                          5 * cd, g[:, 0], beta[:, 0].contiguous(), y[:, 0], dims_of(shape, 5),
                          1 / math.sqrt(d))
    normed = torch.empty(1, 5, 1, d, device="cuda")
    gdn.gated_norm(y, dev["norm_w"], dev["z"], normed, 5, 1, d)
    gk = torch.empty(1, 5, 1, device="cuda")
    gdn.decay_gate(dev["alpha"], dev["dt"], dev["A_log"], gk, 5, 1)
    expect_clean("standalone parts")
    print("checked build clean")


if __name__ == "__main__":
    main()
