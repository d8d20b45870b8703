"""GPU parity of the decode-side entry points against the fp64 oracle, and the
bitwise invariants between them (verify vs decode, commit vs one step,
scan vs steps, fused vs standalone)."""
import math

import numpy as np
import pytest

from gated_delta_ssm_gb300 import synth
from tests._util import (check_out, OUT_TOL, STATE_TOL, as_f32, device_inputs, dims_of, max_rel, out_rel,
                         params_of, run_oracle, to_dev)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gated_delta_ssm_gb300 as gdn  # noqa: E402


def _decode_tokens(shape, dev, T):
    """Run T single-token decode steps; returns outputs [B][T][Hv][d]."""
    dims = dims_of(shape, rows_per_seq=dev["x"].shape[1])
    prm = params_of(dev)
    B, Hv, d = shape.B, shape.Hv, shape.d
    outs = torch.empty(B, T, Hv, d, device="cuda")
    step_out = torch.empty(B, Hv, d, device="cuda")
    for t in range(T):
        gdn.decode_step(dev["state"], dev["hist"], dev["x"][:, t], dev["z"][:, t],
                        dev["alpha"][:, t], dev["beta_logit"][:, t], prm, step_out, dims)
        outs[:, t] = step_out
    torch.cuda.synchronize()
    return outs


# ------------------------------------------------------------------ workload parity
def test_tiny_sequential_16_steps_matches_oracle():
    shape = synth.WORKLOADS["tiny_seq"]
    inp = synth.make_inputs(shape, seed=0)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    outs = _decode_tokens(shape, dev, shape.T).cpu().numpy()
    check_out(outs, ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert max_rel(dev["hist"].cpu().numpy(), ref["hist"], 2) == 0.0


@pytest.mark.parametrize("name", ["decode_b1", "decode_b64"])
def test_single_step_workloads_match_oracle(name):
    shape = synth.WORKLOADS[name]
    inp = synth.make_inputs(shape, seed=1 if name == "decode_b1" else 2)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    out = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    gdn.decode_step(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                    dev["beta_logit"], params_of(dev), out, dims_of(shape))
    torch.cuda.synchronize()
    check_out(out.cpu().numpy(), ref["out"][:, 0])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert max_rel(dev["hist"].cpu().numpy(), ref["hist"], 2) == 0.0


def test_decode_b1_sixteen_steps_state():
    shape = synth.Shape(B=1, T=16, Hq=16, Hv=32, warm=True)
    inp = synth.make_inputs(shape, seed=7)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    outs = _decode_tokens(shape, dev, 16).cpu().numpy()
    check_out(outs, ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL


@pytest.mark.parametrize("W,Hq,Hv,B", [(2, 1, 1, 3), (8, 2, 2, 2), (3, 1, 3, 5), (4, 1, 8, 2),
                                       (5, 2, 8, 1)])
def test_edge_shapes_match_oracle(W, Hq, Hv, B):
    shape = synth.Shape(B=B, T=3, Hq=Hq, Hv=Hv, W=W, warm=True)
    inp = synth.make_inputs(shape, seed=100 + W)
    ref = run_oracle(shape, inp)
    dev = device_inputs(shape, inp)
    outs = _decode_tokens(shape, dev, 3).cpu().numpy()
    check_out(outs, ref["out"])
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert max_rel(dev["hist"].cpu().numpy(), ref["hist"], 2) == 0.0


# ------------------------------------------------------------------ verify K=2 + commit
def test_verify_k2_matches_oracle_and_decode_bitwise():
    shape = synth.WORKLOADS["verify_k2"]
    inp = synth.make_inputs(shape, seed=3)
    ref = run_oracle(shape, inp, snap_after=0)
    dev = device_inputs(shape, inp)
    dims, prm = dims_of(shape), params_of(dev)
    B, Hv, d = shape.B, shape.Hv, shape.d
    st0, hi0 = dev["state"].clone(), dev["hist"].clone()
    snap = torch.empty_like(dev["state"])
    hsnap = torch.empty_like(dev["hist"])
    out = torch.empty(B, 2, Hv, d, device="cuda")
    gdn.verify_k2(dev["state"], dev["hist"], snap, hsnap, dev["x"], dev["z"], dev["alpha"],
                  dev["beta_logit"], prm, out, dims)
    torch.cuda.synchronize()
    # against the oracle
    check_out(out.cpu().numpy(), ref["out"])
    assert max_rel(snap.cpu().numpy(), ref["state_snap"], 2) <= STATE_TOL
    assert max_rel(dev["state"].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert np.array_equal(hsnap.cpu().numpy(), ref["hist_snap"].astype(np.float32))
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))
    # against two single-token decode steps, bit for bit
    dims = dims_of(shape, rows_per_seq=2)
    dec = dict(dev, state=st0.clone(), hist=hi0.clone())
    step = torch.empty(B, Hv, d, device="cuda")
    gdn.decode_step(dec["state"], dec["hist"], dev["x"][:, 0], dev["z"][:, 0], dev["alpha"][:, 0],
                    dev["beta_logit"][:, 0], prm, step, dims)
    torch.cuda.synchronize()
    assert torch.equal(step, out[:, 0])
    assert torch.equal(dec["state"], snap) and torch.equal(dec["hist"], hsnap)
    gdn.decode_step(dec["state"], dec["hist"], dev["x"][:, 1], dev["z"][:, 1], dev["alpha"][:, 1],
                    dev["beta_logit"][:, 1], prm, step, dims)
    torch.cuda.synchronize()
    assert torch.equal(step, out[:, 1])
    assert torch.equal(dec["state"], dev["state"]) and torch.equal(dec["hist"], dev["hist"])
    # commit: accept 1 rolls back to the one-step state, accept 2 keeps both
    acc = dev["accept"]
    gdn.verify_commit(dev["state"], dev["hist"], snap, hsnap, acc, dims_of(shape))
    torch.cuda.synchronize()
    one = (acc == 1).cpu().numpy()
    assert one.any() and (~one).any()
    want_state = torch.where(torch.from_numpy(one).cuda()[:, None, None, None], snap, dec["state"])
    want_hist = torch.where(torch.from_numpy(one).cuda()[:, None, None], hsnap, dec["hist"])
    assert torch.equal(dev["state"], want_state)
    assert torch.equal(dev["hist"], want_hist)


def test_commit_flags_other_accept_values_and_leaves_them_unchanged():
    shape = synth.Shape(B=4, T=2, Hq=1, Hv=2, warm=True)
    inp = synth.make_inputs(shape, seed=9)
    dev = device_inputs(shape, inp)
    snap = torch.zeros_like(dev["state"])
    hsnap = torch.zeros_like(dev["hist"])
    before = dev["state"].clone(), dev["hist"].clone()
    assert gdn.check_device() == 0
    # 2 is a valid count (keep both positions); 0, 3 and -1 are out of range
    acc = torch.tensor([0, 2, 3, -1], dtype=torch.int32, device="cuda")
    gdn.verify_commit(dev["state"], dev["hist"], snap, hsnap, acc, dims_of(shape))
    assert gdn.check_device() == 16
    assert torch.equal(dev["state"], before[0]) and torch.equal(dev["hist"], before[1])
    # valid counts only: nothing flagged
    acc = torch.tensor([2, 2, 2, 2], dtype=torch.int32, device="cuda")
    gdn.verify_commit(dev["state"], dev["hist"], snap, hsnap, acc, dims_of(shape))
    assert gdn.check_device() == 0


# ------------------------------------------------------------------ standalone parts
def test_standalone_parts_match_oracle_and_fused():
    shape = synth.Shape(B=3, T=1, Hq=4, Hv=8, warm=True)
    inp = synth.make_inputs(shape, seed=21)
    ref = run_oracle(shape, inp, intermediates=True)
    dev = device_inputs(shape, inp)
    dims = dims_of(shape)
    B, Hq, Hv, d, cd = shape.B, shape.Hq, shape.Hv, shape.d, shape.conv_dim
    # conv + SiLU + L2
    hist = dev["hist"].clone()
    conv = torch.empty(B, 1, cd, device="cuda")
    gdn.conv_update(hist, dev["x"], dev["conv_w"], conv, dims, 1, 1e-6)
    # gate
    g = torch.empty(B, Hv, device="cuda")
    gdn.decay_gate(dev["alpha"], dev["dt"], dev["A_log"], g, B, Hv)
    torch.cuda.synchronize()
    assert max_rel(conv.cpu().numpy(), ref["conv"], 1) <= 1e-5
    assert np.array_equal(hist.cpu().numpy(), ref["hist"].astype(np.float32))
    assert max_rel(g.cpu().numpy(), ref["g"][:, 0], 1) <= 1e-5
    # recurrence fed the GPU conv + gate outputs, beta from torch
    beta = torch.sigmoid(dev["beta_logit"][:, 0].float()).contiguous()
    state = dev["state"].clone()
    y = torch.empty(B, Hv, d, device="cuda")
    c0 = conv[:, 0]
    gdn.recurrence_decode(state, c0, c0[:, Hq * d:], c0[:, 2 * Hq * d:], cd, g, beta, y, dims,
                          1 / math.sqrt(d))
    out = torch.empty_like(y)
    gdn.gated_norm(y, dev["norm_w"], dev["z"][:, 0], out, B, Hv, d, Hv * d, 1e-6)
    torch.cuda.synchronize()
    check_out(y.cpu().numpy(), ref["y"][:, 0])
    check_out(out.cpu().numpy(), ref["out"][:, 0])
    assert max_rel(state.cpu().numpy(), ref["state"], 2) <= STATE_TOL
    # the fused step agrees with the composition (beta differs only in its sigmoid rounding)
    fused = torch.empty_like(y)
    fstate = dev["state"].clone()
    fhist = dev["hist"].clone()
    gdn.decode_step(fstate, fhist, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                    params_of(dev), fused, dims)
    torch.cuda.synchronize()
    assert torch.equal(fhist, hist)
    assert max_rel(fused.cpu().numpy(), out.cpu().numpy(), 1) <= 1e-5
    assert max_rel(fstate.cpu().numpy(), state.cpu().numpy(), 2) <= 1e-5


def test_recurrence_fed_oracle_inputs():
    # the recurrence alone, fed the oracle's own prepared q^, k^, v, g, beta (fp32-rounded)
    shape = synth.Shape(B=2, T=1, Hq=2, Hv=6, warm=True)
    inp = synth.make_inputs(shape, seed=22)
    ref = run_oracle(shape, inp, intermediates=True)
    B, Hq, Hv, d, cd = shape.B, shape.Hq, shape.Hv, shape.d, shape.conv_dim
    conv = to_dev(ref["conv"][:, 0].astype(np.float32))
    g = to_dev(ref["g"][:, 0].astype(np.float32))
    beta = to_dev(ref["beta"][:, 0].astype(np.float32))
    state = to_dev(inp["state"])
    y = torch.empty(B, Hv, d, device="cuda")
    gdn.recurrence_decode(state, conv, conv[:, Hq * d:], conv[:, 2 * Hq * d:], cd, g, beta, y,
                          dims_of(shape), 1 / math.sqrt(d))
    torch.cuda.synchronize()
    assert max_rel(y.cpu().numpy(), ref["y"][:, 0], 1) <= 1e-4
    assert max_rel(state.cpu().numpy(), ref["state"], 2) <= 1e-5


def test_gated_norm_aliases_and_bf16_z():
    shape = synth.Shape(B=5, T=1, Hq=1, Hv=4, warm=True)
    inp = synth.make_inputs(shape, seed=23)
    ref = run_oracle(shape, inp, intermediates=True)
    y = to_dev(ref["y"][:, 0].astype(np.float32))
    z = to_dev(inp["z"][:, 0], "bf16")
    w = to_dev(inp["norm_w"])
    gdn.gated_norm(y, w, z, y, shape.B, shape.Hv, 128, shape.Hv * 128, 1e-6)   # in place
    torch.cuda.synchronize()
    assert max_rel(y.cpu().numpy(), ref["out"][:, 0], 1) <= 1e-5


def test_conv_scan_equals_single_steps_bitwise():
    shape = synth.Shape(B=2, T=7, Hq=2, Hv=4, W=4, warm=True)
    inp = synth.make_inputs(shape, seed=24)
    dev = device_inputs(shape, inp)
    dims = dims_of(shape)
    cd = shape.conv_dim
    h1 = dev["hist"].clone()
    full = torch.empty(shape.B, shape.T, cd, device="cuda")
    gdn.conv_update(h1, dev["x"], dev["conv_w"], full, dims, shape.T, 1e-6)
    h2 = dev["hist"].clone()
    steps = torch.empty_like(full)
    one = torch.empty(shape.B, 1, cd, device="cuda")
    for t in range(shape.T):
        xt = dev["x"][:, t:t + 1].contiguous()
        gdn.conv_update(h2, xt, dev["conv_w"], one, dims, 1, 1e-6)
        steps[:, t] = one[:, 0]
    torch.cuda.synchronize()
    assert torch.equal(full, steps) and torch.equal(h1, h2)
    ref = run_oracle(shape, inp, intermediates=True)
    assert max_rel(full.cpu().numpy(), ref["conv"], 1) <= 1e-5


@pytest.mark.parametrize("B,T,W,act,pad", [(2, 100, 4, "bf16", 0), (1, 33, 8, "f32", 0),
                                           (3, 64, 2, "bf16", 0), (2, 3, 8, "bf16", 0),
                                           (2, 200, 4, "f32", 0), (2, 100, 4, "bf16", 4),
                                           (1, 70, 3, "f32", 1)])
def test_token_parallel_conv_equals_serial_steps(B, T, W, act, pad):
    # several tiles with a ragged tail (and T < W-1): the multi-token kernels against
    # T single-token calls of the serial kernel, bit for bit. Rows padded by a
    # non-multiple of 16 bytes take the plain-load kernel instead of the tiled one.
    base = synth.Shape(B=B, T=T, Hq=2, Hv=6, W=W, act_dtype=act, warm=True)
    shape = synth.Shape(B=B, T=T, Hq=2, Hv=6, W=W, act_dtype=act, warm=True,
                        x_stride=base.conv_dim + pad)
    inp = synth.make_inputs(shape, seed=27 + T)
    dev = device_inputs(shape, inp)
    dims = dims_of(shape)
    cd = shape.conv_dim
    h1 = dev["hist"].clone()
    full = torch.empty(B, T, cd, device="cuda")
    gdn.conv_update(h1, dev["x"], dev["conv_w"], full, dims, T, 1e-6)
    h2 = dev["hist"].clone()
    steps = torch.empty_like(full)
    one = torch.empty(B, 1, cd, device="cuda")
    dims1 = dims_of(shape, rows_per_seq=T)
    for t in range(T):
        gdn.conv_update(h2, dev["x"][:, t:t + 1], dev["conv_w"], one, dims1, 1, 1e-6)
        steps[:, t] = one[:, 0]
    torch.cuda.synchronize()
    assert torch.equal(full, steps) and torch.equal(h1, h2)
    ref = run_oracle(shape, inp, intermediates=True)
    assert max_rel(full.cpu().numpy(), ref["conv"], 1) <= 1e-5
    assert np.array_equal(h1.cpu().numpy(), ref["hist"].astype(np.float32))


def test_token_parallel_conv_full_prefill_size_equals_serial():
    # 4 x 8192 tokens of the 8192-channel prefill layer, every element
    shape = synth.WORKLOADS["prefill"]
    inp = synth.make_inputs(shape, seed=28)
    dev = device_inputs(shape, inp)
    B, T, cd = shape.B, shape.T, shape.conv_dim
    h1 = dev["hist"].clone()
    full = torch.empty(B, T, cd, device="cuda")
    gdn.conv_update(h1, dev["x"], dev["conv_w"], full, dims_of(shape), T, 1e-6)
    h2 = dev["hist"].clone()
    one = torch.empty(B, 1, cd, device="cuda")
    dims1 = dims_of(shape, rows_per_seq=T)
    same = True
    for t in range(T):
        gdn.conv_update(h2, dev["x"][:, t:t + 1], dev["conv_w"], one, dims1, 1, 1e-6)
        same &= bool(torch.equal(one[:, 0], full[:, t]))
    torch.cuda.synchronize()
    assert same and torch.equal(h1, h2)


# ------------------------------------------------------------------ bf16-state decode
def _bf16_state(inp):
    """The workload's state rounded to bf16: (bf16 bits, exact float32 values)."""
    bits = synth.bf16_round(inp["state"])
    return bits, synth.bf16_to_f32(bits)


def test_bf16_state_step_is_the_float_step_rounded():
    # same inputs, state values exactly bf16: the bf16-state kernel stores exactly
    # the round-to-nearest-even of what the float32 kernel computes
    shape = synth.WORKLOADS["decode_b64"]
    inp = synth.make_inputs(shape, seed=29)
    dev = device_inputs(shape, inp)
    bits, f32 = _bf16_state(inp)
    st16 = to_dev(bits, "bf16")
    st32 = to_dev(f32)
    h16, h32 = dev["hist"].clone(), dev["hist"].clone()
    out16 = torch.empty(shape.B, shape.Hv, shape.d, device="cuda", dtype=torch.bfloat16)
    out32 = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    gdn.decode_step_bf16_state(st16, h16, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                               params_of(dev), out16, dims_of(shape))
    gdn.decode_step(st32, h32, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                    params_of(dev), out32, dims_of(shape))
    torch.cuda.synchronize()
    assert torch.equal(st16, st32.to(torch.bfloat16))
    assert torch.equal(out16, out32.to(torch.bfloat16))
    assert torch.equal(h16, h32)


@pytest.mark.parametrize("name,steps,seed", [("decode_b1", 8, 30), ("tiny_seq", 16, 31),
                                             ("verify_k2", 2, 32)])
def test_bf16_state_decode_matches_rounded_oracle(name, steps, seed):
    # against the oracle's bf16-state variant (state and outputs rounded to bf16
    # after every step). A stored value is the RNE of a float32 result within
    # ~1e-6 of the oracle's fp64 one, so the two roundings differ by at most one
    # bf16 ulp (2^-8 relative), and a flipped state entry perturbs later steps
    # by about as much again: 2^-7 normwise for state and outputs.
    base = synth.WORKLOADS[name]
    shape = synth.Shape(B=base.B, T=steps, Hq=base.Hq, Hv=base.Hv, act_dtype=base.act_dtype,
                        warm=True)
    inp = synth.make_inputs(shape, seed=seed)
    bits, f32 = _bf16_state(inp)
    ref = run_oracle(shape, dict(inp, state=f32), bf16_state=True)
    dev = device_inputs(shape, inp)
    st = to_dev(bits, "bf16")
    dims = dims_of(shape, rows_per_seq=steps)
    outs = torch.empty(shape.B, steps, shape.Hv, shape.d, device="cuda", dtype=torch.bfloat16)
    one = torch.empty(shape.B, shape.Hv, shape.d, device="cuda", dtype=torch.bfloat16)
    for t in range(steps):
        gdn.decode_step_bf16_state(st, dev["hist"], dev["x"][:, t], dev["z"][:, t],
                                   dev["alpha"][:, t], dev["beta_logit"][:, t], params_of(dev),
                                   one, dims)
        outs[:, t] = one
    torch.cuda.synchronize()
    tol = 2.0 ** -7
    check_out(outs.float().cpu().numpy(), ref["out"], tol)
    assert max_rel(st.float().cpu().numpy(), ref["state"], 2) <= tol
    assert np.array_equal(dev["hist"].cpu().numpy(), ref["hist"].astype(np.float32))


def test_result_independent_of_batch_split():
    # the same sequence decoded alone (few CTAs: row-split clusters) and inside a
    # large batch (one CTA per head) gives identical bits
    big = synth.Shape(B=64, T=1, Hq=16, Hv=32, warm=True)
    inp = synth.make_inputs(big, seed=25)
    dev = device_inputs(big, inp)
    out_big = torch.empty(64, 32, 128, device="cuda")
    st_big = dev["state"].clone()
    gdn.decode_step(st_big, dev["hist"].clone(), dev["x"], dev["z"], dev["alpha"],
                    dev["beta_logit"], params_of(dev), out_big, dims_of(big))
    small = synth.Shape(B=1, T=1, Hq=16, Hv=32, warm=True)
    b = 17
    st1 = dev["state"][b:b + 1].clone()
    out1 = torch.empty(1, 32, 128, device="cuda")
    gdn.decode_step(st1, dev["hist"][b:b + 1].clone(), dev["x"][b:b + 1], dev["z"][b:b + 1],
                    dev["alpha"][b:b + 1], dev["beta_logit"][b:b + 1], params_of(dev), out1,
                    dims_of(small))
    torch.cuda.synchronize()
    assert torch.equal(out1[0], out_big[b])
    assert torch.equal(st1[0], st_big[b])


def test_decode_at_the_largest_batch():
    # n_seq = 65535, the largest the entry points accept (one CTA row per sequence);
    # the first, a middle and the last sequence are held to the oracle
    shape = synth.Shape(B=65535, T=1, Hq=1, Hv=1, warm=False)
    inp = synth.make_inputs(shape, seed=36)
    dev = device_inputs(shape, inp)
    out = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
    gdn.decode_step(dev["state"], dev["hist"], dev["x"], dev["z"], dev["alpha"],
                    dev["beta_logit"], params_of(dev), out, dims_of(shape))
    torch.cuda.synchronize()
    seqs = [0, 32767, 65534]
    ref = run_oracle(shape, inp, seqs=seqs)
    check_out(out.cpu().numpy()[seqs], ref["out"][:, 0])
    assert max_rel(dev["state"][seqs].cpu().numpy(), ref["state"], 2) <= STATE_TOL
    assert np.array_equal(dev["hist"][seqs].cpu().numpy(), ref["hist"].astype(np.float32))


def test_repeat_runs_are_deterministic():
    shape = synth.WORKLOADS["decode_b64"]
    inp = synth.make_inputs(shape, seed=26)
    dev = device_inputs(shape, inp)
    res = []
    for _ in range(2):
        st, hi = dev["state"].clone(), dev["hist"].clone()
        out = torch.empty(shape.B, shape.Hv, shape.d, device="cuda")
        gdn.decode_step(st, hi, dev["x"], dev["z"], dev["alpha"], dev["beta_logit"],
                        params_of(dev), out, dims_of(shape))
        torch.cuda.synchronize()
        res.append((out, st, hi))
    assert all(torch.equal(a, b) for a, b in zip(res[0], res[1]))


@pytest.mark.parametrize("n_first", [64, 8])
def test_step_reads_inputs_the_previous_step_just_wrote(n_first):
    """The decode launch is a programmatic dependent of the kernel before it in the
    stream, and the decode kernel lets its dependents start before its outputs are
    written (a launch of one wave or less as soon as its own grid wait returns, a
    larger one once its state stores are issued: 64 sequences here give 1024 CTAs,
    8 give 128). A step whose x and z rows ARE the output of the step just before it
    must still read them only once that step is done: the same bits as with a device
    synchronisation between the two calls. The first step's output buffer starts as
    NaN, so a read that came too early would show."""
    big = synth.Shape(B=n_first, T=1, Hq=4, Hv=8, act_dtype="f32", warm=True)
    inp1 = synth.make_inputs(big, seed=140)
    dev1 = device_inputs(big, inp1)
    # the second step: a quarter as many sequences, whose fp32 x rows (x then z in
    # one row) are carved out of the first step's [B][8][128] output
    small = synth.Shape(B=n_first // 4, T=1, Hq=4, Hv=8, act_dtype="f32", warm=True)
    row = 2 * small.conv_dim
    assert small.B * row <= big.B * big.Hv * big.d
    inp2 = synth.make_inputs(small, seed=141)
    dev2 = device_inputs(small, inp2)
    dims2 = gdn.Dims(n_seq=small.B, n_qk_heads=small.Hq, n_v_heads=small.Hv, head_dim=small.d,
                     d_conv=small.W, x_stride=row, z_stride=row, gate_stride=small.Hv)
    results = []
    for sync in (False, True):
        st1, hi1 = dev1["state"].clone(), dev1["hist"].clone()
        st2, hi2 = dev2["state"].clone(), dev2["hist"].clone()
        out1 = torch.full((big.B, big.Hv, big.d), float("nan"), device="cuda")
        out2 = torch.empty(small.B, small.Hv, small.d, device="cuda")
        rows = out1.view(-1)[:small.B * row].view(small.B, row)
        torch.cuda.synchronize()
        gdn.decode_step(st1, hi1, dev1["x"][:, 0], dev1["z"][:, 0], dev1["alpha"][:, 0],
                        dev1["beta_logit"][:, 0], params_of(dev1), out1, dims_of(big))
        if sync:
            torch.cuda.synchronize()
        gdn.decode_step(st2, hi2, rows, rows[:, small.conv_dim:], dev2["alpha"][:, 0],
                        dev2["beta_logit"][:, 0], params_of(dev2), out2, dims2)
        torch.cuda.synchronize()
        results.append((out2, st2, hi2))
    assert gdn.check_device() == 0
    assert torch.isfinite(results[1][0]).all()
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a, b)


def test_back_to_back_steps_on_one_state_equal_synchronised_steps():
    """Single-sequence steps (one wave: each launch prefetches its state rows into L2
    and makes the next launch resident before its own work) stepping the SAME state
    and conv history 24 times in a row give the bits of the same steps with a device
    synchronisation after each."""
    shape = synth.WORKLOADS["decode_b1"]
    inp = synth.make_inputs(shape, seed=142)
    dev = device_inputs(shape, inp)
    res = []
    for sync in (False, True):
        st, hi = dev["state"].clone(), dev["hist"].clone()
        outs = torch.full((24, shape.B, shape.Hv, shape.d), float("nan"), device="cuda")
        torch.cuda.synchronize()
        for i in range(24):
            gdn.decode_step(st, hi, dev["x"][:, 0], dev["z"][:, 0], dev["alpha"][:, 0],
                            dev["beta_logit"][:, 0], params_of(dev), outs[i], dims_of(shape))
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        res.append((outs, st, hi))
    assert gdn.check_device() == 0
    assert torch.isfinite(res[1][0]).all()
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
