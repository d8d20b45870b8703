"""GPU parity of the token-serial entry points: the recurrence scan, the fused
layer scan and the generic-K draft verification with its commit.

Each is held to the fp64 oracle and, bit for bit, to the single-step entry
points it is defined to equal (n decode steps; verify_k2 at K = 2). The layer
scan then serves as the on-device sequential reference for the chunked
prefill at the full 4 x 8192 size."""
import math

import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import (check_out, OUT_TOL, STATE_TOL, device_inputs, dims_of, max_rel, out_rel, params_of,
                         run_oracle, to_dev)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402


def _steps(shape, dev, state, hist, T, snaps=False):
    """T single-token gdn_decode_step calls from (state, hist), in place.
    Returns outputs [B][T][Hv][d] and, with snaps, the (state, hist) after each token."""
    dims = dims_of(shape, rows_per_seq=dev["x"].shape[1])
    prm = params_of(dev)
    outs = torch.empty(shape.B, T, shape.Hv, shape.d, device="cuda")
    one = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    after = []
    for t in range(T):
        gdn.decode_step(state, hist, dev["x"][:, t], dev["z"][:, t], dev["alpha"][:, t],
                        dev["beta_logit"][:, t], prm, one, dims)
        outs[:, t] = one
        if snaps:
            after.append((state.clone(), hist.clone()))
    torch.cuda.synchronize()
    return outs, after


def _layer_scan(shape, dev, T):
    out = torch.empty(shape.B, T, shape.Hv, shape.d, device="cuda")
    gdn.layer_scan(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                   params_of(dev), out, dims_of(shape), T)
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------ layer scan
# (B, Hq, Hv, W, act): the launch picks 1, 2 or 4 row slices per head from B * Hv
@pytest.mark.parametrize("B,Hq,Hv,W,act", [(1, 1, 4, 4, "bf16"), (4, 16, 32, 4, "bf16"),
                                           (12, 4, 32, 4, "f32"), (3, 2, 6, 3, "bf16"),
                                           (2, 1, 8, 2, "f32"), (2, 2, 2, 8, "bf16")])
def test_layer_scan_equals_decode_steps_bitwise(B, Hq, Hv, W, act):
    shape = synth.Shape(B=B, T=9, Hq=Hq, Hv=Hv, W=W, act_dtype=act, warm=True)
    inp = synth.make_inputs(shape, seed=40 + B + W)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    out = _layer_scan(shape, dev, shape.T)
    ref_out, _ = _steps(shape, dev, st, hi, shape.T)
    assert torch.equal(out, ref_out)
    assert torch.equal(dev["state"], st)
    assert torch.equal(dev["hist"], hi)


@pytest.mark.parametrize("name,seed", [("tiny_seq", 41), ("ragged", 42)])
def test_layer_scan_matches_oracle(name, seed):
    shape = (synth.WORKLOADS["tiny_seq"] if name == "tiny_seq"
             else synth.Shape(B=3, T=37, Hq=2, Hv=6, W=4, warm=False))
    inp = synth.make_inputs(shape, seed=seed)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    out = _layer_scan(shape, dev, shape.T).cpu().numpy()
    check_out(out, ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


def test_chunked_prefill_full_size_against_layer_scan():
    # the full 4 x 8192 prefill workload, every output token compared with the
    # token-serial scan (itself equal to 8192 decode steps bit for bit)
    shape = synth.WORKLOADS["prefill"]
    inp = synth.make_inputs(shape, seed=43)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    seq = _layer_scan(shape, dev, shape.T)
    chk = torch.empty_like(seq)
    gdn.prefill_chunked(st, hi, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                        params_of(dev), chk, dims_of(shape), shape.T, 64)
    torch.cuda.synchronize()
    # normwise per (sequence, V head) slice, computed on the device in float64
    num = (chk.double() - seq.double()).abs().amax(dim=(1, 3))
    den = seq.double().abs().amax(dim=(1, 3)).clamp_min(1e-300)
    assert float((num / den).max()) <= OUT_TOL
    assert max_rel(st.cpu().numpy(), dev["state"].cpu().numpy(), 2) <= STATE_TOL
    assert torch.equal(hi, dev["hist"])


# ------------------------------------------------------------------ verify K + commit
def _verify(shape, dev, K):
    B, Hv, d = shape.B, shape.Hv, shape.d
    ssnap = torch.full((B, max(K - 1, 1), Hv, d, d), float("nan"), device="cuda")
    csnap = torch.full((B, K) + tuple(dev["hist"].shape[1:]), float("nan"), device="cuda")
    out = torch.empty(B, K, Hv, d, device="cuda")
    gdn.verify_kn(dev["state"], dev["hist"], ssnap, csnap, dev["x"], dev["z"], dev["alpha"],
                  dev["beta_logit"], params_of(dev), out, dims_of(shape), K)
    torch.cuda.synchronize()
    return out, ssnap, csnap


@pytest.mark.parametrize("K,B,Hq,Hv,act", [(1, 2, 2, 4, "bf16"), (3, 3, 2, 4, "bf16"),
                                           (5, 2, 1, 3, "f32"), (17, 2, 2, 4, "bf16"),
                                           (4, 40, 16, 32, "bf16")])
def test_verify_kn_equals_decode_steps_and_oracle(K, B, Hq, Hv, act):
    shape = synth.Shape(B=B, T=K, Hq=Hq, Hv=Hv, act_dtype=act, warm=True)
    inp = synth.make_inputs(shape, seed=50 + K)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    out, ssnap, csnap = _verify(shape, dev, K)
    # bit for bit against K decode steps, snapshot by snapshot
    ref_out, after = _steps(shape, dev, st, hi, K, snaps=True)
    assert torch.equal(out, ref_out)
    assert torch.equal(dev["state"], st) and torch.equal(dev["hist"], hi)
    for p in range(K):
        assert torch.equal(csnap[:, p], after[p][1])
        if p < K - 1:
            assert torch.equal(ssnap[:, p], after[p][0])
    # against the oracle: outputs, committed state, and each state snapshot
    seqs = None if B <= 4 else [0, B // 2, B - 1]
    ref = run_oracle(shape, inp, seqs=seqs)
    pick = slice(None) if seqs is None else seqs
    check_out(out.cpu().numpy()[pick], ref["out"])
    assert max_rel(dev["state"].cpu().numpy()[pick], ref["state"], 2) <= STATE_TOL
    if K > 1 and seqs is None:
        mid = K // 2
        part = run_oracle(shape, inp, T=mid + 1)
        assert max_rel(ssnap[:, mid].cpu().numpy(), part["state"], 2) <= STATE_TOL
        assert np.array_equal(csnap[:, mid].cpu().numpy(), part["hist"].astype(np.float32))


@pytest.mark.parametrize("K,B,Hq,Hv,W,act", [(4, 1, 1, 8, 8, "f32"), (3, 2, 2, 2, 2, "bf16"),
                                             (2, 5, 1, 4, 5, "bf16"), (4, 3, 2, 4, 3, "f32"),
                                             (8, 1, 1, 8, 8, "f32"), (6, 2, 2, 2, 2, "bf16"),
                                             (5, 3, 2, 4, 3, "f32"), (7, 40, 2, 8, 4, "bf16")])
def test_verify_kn_fused_edge_shapes_equal_decode_steps(K, B, Hq, Hv, W, act):
    # drafts of up to eight positions run in the fused step kernel: conv windows of 2..8
    # taps, eight V heads per QK head, one sequence (row slices and clusters), and a
    # batch of whole heads (K = 7, 40 sequences)
    shape = synth.Shape(B=B, T=K, Hq=Hq, Hv=Hv, W=W, act_dtype=act, warm=True)
    inp = synth.make_inputs(shape, seed=70 + 10 * K + W)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    out, ssnap, csnap = _verify(shape, dev, K)
    ref_out, after = _steps(shape, dev, st, hi, K, snaps=True)
    assert gdn.check_device() == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(dev["state"], st) and torch.equal(dev["hist"], hi)
    for p in range(K):
        assert torch.equal(csnap[:, p], after[p][1])
        if p < K - 1:
            assert torch.equal(ssnap[:, p], after[p][0])
    ref = run_oracle(shape, inp)
    check_out(out.cpu().numpy(), ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL


def test_verify_kn_at_k2_equals_verify_k2_bitwise():
    shape = synth.WORKLOADS["verify_k2"]
    inp = synth.make_inputs(shape, seed=60)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    out, ssnap, csnap = _verify(shape, dev, 2)
    snap2, hsnap2 = torch.empty_like(st), torch.empty_like(hi)
    out2 = torch.empty_like(out)
    gdn.verify_k2(st, hi, snap2, hsnap2, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                  params_of(dev), out2, dims_of(shape))
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
    assert torch.equal(dev["state"], st) and torch.equal(dev["hist"], hi)
    assert torch.equal(ssnap[:, 0], snap2) and torch.equal(csnap[:, 0], hsnap2)
    assert torch.equal(csnap[:, 1], hi)


def test_commit_kn_restores_the_accepted_prefix():
    K = 6
    shape = synth.Shape(B=8, T=K, Hq=2, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=61)
    dev = device_inputs(shape, inp)
    st, hi = dev["state"].clone(), dev["hist"].clone()
    _, ssnap, csnap = _verify(shape, dev, K)
    _, after = _steps(shape, dev, st, hi, K, snaps=True)
    n = torch.tensor([1, 2, 3, 4, 5, 6, 1, 6], dtype=torch.int32, device="cuda")
    gdn.verify_commit_kn(dev["state"], dev["hist"], ssnap, csnap, n, dims_of(shape), K)
    torch.cuda.synchronize()
    assert gdn.check_device() == 0
    for b, nb in enumerate(n.tolist()):
        assert torch.equal(dev["state"][b], after[nb - 1][0][b])
        assert torch.equal(dev["hist"][b], after[nb - 1][1][b])


def test_commit_kn_flags_out_of_range_counts():
    K = 3
    shape = synth.Shape(B=4, T=K, Hq=1, Hv=2, warm=True)
    inp = synth.make_inputs(shape, seed=62)
    dev = device_inputs(shape, inp)
    _, ssnap, csnap = _verify(shape, dev, K)
    before = dev["state"].clone(), dev["hist"].clone()
    n = torch.tensor([0, 4, -1, 3], dtype=torch.int32, device="cuda")
    assert gdn.check_device() == 0
    gdn.verify_commit_kn(dev["state"], dev["hist"], ssnap, csnap, n, dims_of(shape), K)
    assert gdn.check_device() == 16
    assert gdn.check_device() == 0          # read and cleared
    assert torch.equal(dev["state"], before[0]) and torch.equal(dev["hist"], before[1])


# ------------------------------------------------------------------ recurrence scan
@pytest.mark.parametrize("B,Hq,Hv,T", [(2, 2, 4, 11), (1, 1, 1, 5), (6, 4, 32, 3)])
def test_recurrence_scan_equals_decode_calls_and_oracle(B, Hq, Hv, T):
    shape = synth.Shape(B=B, T=T, Hq=Hq, Hv=Hv, warm=True)
    inp = synth.make_inputs(shape, seed=70 + T)
    ref = run_oracle(shape, inp, intermediates=True)
    d, cd = shape.d, shape.conv_dim
    # the oracle's prepared operands, rounded to float32
    conv = to_dev(ref["conv"].astype(np.float32))          # [B][T][cd]
    g = to_dev(ref["g"].astype(np.float32))                # [B][T][Hv]
    beta = to_dev(ref["beta"].astype(np.float32))
    scale = 1 / math.sqrt(d)
    state = to_dev(inp["state"])
    y = torch.empty(B, T, Hv, d, device="cuda")
    dims = dims_of(shape)
    gdn.recurrence_scan(state, conv, conv[..., Hq * d:], conv[..., 2 * Hq * d:], cd, g, beta, y,
                        dims, T, scale)
    # T single-step calls over token slices (rows T*cd apart)
    st2 = to_dev(inp["state"])
    y2 = torch.empty_like(y)
    one = torch.empty(B, Hv, d, device="cuda")
    for t in range(T):
        ct = conv[:, t]
        gdn.recurrence_decode(st2, ct, ct[:, Hq * d:], ct[:, 2 * Hq * d:], T * cd,
                              g[:, t].contiguous(), beta[:, t].contiguous(), one, dims, scale)
        y2[:, t] = one
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(state, st2)
    assert max_rel(y.cpu().numpy(), ref["y"], 1) <= 1e-4
    assert max_rel(state.cpu().numpy(), ref["state"], 2) <= 1e-5
