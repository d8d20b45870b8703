"""Pins for the oracle's whole-layer wiring (CPU only).

The per-part pins live in test_oracle_pins.py. Here the composition is held
to an independent numpy restatement of the wiring (split of the conv output
into [Q | K | V], L2 on Q and K only, GQA map h -> h // r, gated norm per
V head), built from the separately pinned parts, plus the snapshot and
scan-equals-steps properties.
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle
from gated_delta_ssm_gb300 import synth


def _small(B=2, T=5, Hq=2, Hv=4, d=16, W=4, warm=True, seed=3):
    shape = synth.Shape(B=B, T=T, Hq=Hq, Hv=Hv, d=d, W=W, act_dtype="f32", warm=warm)
    return shape, synth.make_inputs(shape, seed)


def _run(shape, inp, **kw):
    return oracle.layer(inp["x"], inp["z"], inp["alpha"], inp["beta_logit"], inp["conv_w"],
                        inp["dt"], inp["A_log"], inp["norm_w"], inp["state"], inp["hist"],
                        Hq=shape.Hq, W=shape.W, **kw)


def test_layer_matches_numpy_wiring():
    shape, inp = _small()
    res = _run(shape, inp, intermediates=True)
    d, Hq, Hv, W = shape.d, shape.Hq, shape.Hv, shape.W
    r = Hv // Hq
    for b in range(shape.B):
        S = np.swapaxes(inp["state"][b].astype(np.float64), -1, -2)    # [h][i][j]
        hist = inp["hist"][b].astype(np.float64)
        for t in range(shape.T):
            x = inp["x"][b, t].astype(np.float64)
            # conv via numpy correlate over [history | x]
            stream = np.concatenate([hist, x[:, None]], 1)
            pre = np.einsum("cw,cw->c", stream, inp["conv_w"].astype(np.float64))
            c = pre * expit(pre)
            hist = stream[:, 1:]
            q = c[:Hq * d].reshape(Hq, d)
            k = c[Hq * d:2 * Hq * d].reshape(Hq, d)
            v = c[2 * Hq * d:].reshape(Hv, d)
            q = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6)
            k = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
            np.testing.assert_allclose(res["conv"][b, t], np.concatenate([q.ravel(), k.ravel(), v.ravel()]),
                                       rtol=1e-12, atol=1e-14)
            sp = np.logaddexp(0, inp["alpha"][b, t].astype(np.float64) + inp["dt"])
            g = -np.exp(inp["A_log"].astype(np.float64)) * sp
            beta = expit(inp["beta_logit"][b, t].astype(np.float64))
            for h in range(Hv):
                kk, qq = k[h // r], q[h // r]
                Snew = math.exp(g[h]) * (np.eye(d) - beta[h] * np.outer(kk, kk)) @ S[h] \
                    + beta[h] * np.outer(kk, v[h])
                S[h] = Snew
                y = Snew.T @ qq / math.sqrt(d)
                np.testing.assert_allclose(res["y"][b, t, h], y, rtol=1e-10, atol=1e-12)
                z = inp["z"][b, t, h * d:(h + 1) * d].astype(np.float64)
                o = y / np.sqrt(np.mean(y * y) + 1e-6) * inp["norm_w"] * z * expit(z)
                np.testing.assert_allclose(res["out"][b, t, h], o, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(res["state"][b], np.swapaxes(S, -1, -2), rtol=1e-10, atol=1e-12)
        np.testing.assert_array_equal(res["hist"][b], hist)


def test_gqa_map_uses_floor_h_over_r():
    # Changing only QK head 1's input channels must leave V heads 0..r-1 untouched.
    shape, inp = _small(B=1, T=3, Hq=2, Hv=6)
    base = _run(shape, inp)
    d = shape.d
    inp2 = dict(inp)
    inp2["x"] = inp["x"].copy()
    inp2["x"][..., 1 * d:2 * d] += 1.0                       # Q head 1
    inp2["x"][..., (2 + 1) * d:(2 + 2) * d] -= 0.5          # K head 1
    alt = _run(shape, inp2)
    np.testing.assert_array_equal(alt["out"][..., :3, :], base["out"][..., :3, :])
    assert np.abs(alt["out"][..., 3:, :] - base["out"][..., 3:, :]).max() > 1e-3


def test_scan_equals_single_steps():
    shape, inp = _small(B=1, T=6)
    full = _run(shape, inp)
    st, hi = inp["state"], inp["hist"]
    outs = []
    for t in range(shape.T):
        step = oracle.layer(inp["x"][:, t:t + 1], inp["z"][:, t:t + 1], inp["alpha"][:, t:t + 1],
                            inp["beta_logit"][:, t:t + 1], inp["conv_w"], inp["dt"], inp["A_log"],
                            inp["norm_w"], st, hi, Hq=shape.Hq, W=shape.W)
        outs.append(step["out"][:, 0])
        st, hi = step["state"], step["hist"]
    np.testing.assert_array_equal(np.stack(outs, 1), full["out"])
    np.testing.assert_array_equal(st, full["state"])
    np.testing.assert_array_equal(hi, full["hist"])


def test_snapshot_is_state_after_first_token():
    shape, inp = _small(B=2, T=2)
    two = _run(shape, inp, snap_after=0)
    one = oracle.layer(inp["x"][:, :1], inp["z"][:, :1], inp["alpha"][:, :1],
                       inp["beta_logit"][:, :1], inp["conv_w"], inp["dt"], inp["A_log"],
                       inp["norm_w"], inp["state"], inp["hist"], Hq=shape.Hq, W=shape.W)
    np.testing.assert_array_equal(two["state_snap"], one["state"])
    np.testing.assert_array_equal(two["hist_snap"], one["hist"])


def test_strided_rows_and_z_inside_row():
    # the batched-decode layout: x rows 2*conv_dim apart, z at offset conv_dim in the row
    base = synth.Shape(B=3, T=1, Hq=2, Hv=6, d=16, act_dtype="f32", warm=True)
    strided = synth.Shape(B=3, T=1, Hq=2, Hv=6, d=16, act_dtype="f32", warm=True,
                          x_stride=2 * base.conv_dim, z_in_x=True)
    a = synth.make_inputs(base, 11)
    b = synth.make_inputs(strided, 11)
    np.testing.assert_array_equal(a["x"], b["x"][..., :base.conv_dim])
    np.testing.assert_array_equal(a["z"], b["z"])
    ra = _run(base, a)
    rb = _run(strided, b)
    np.testing.assert_array_equal(ra["out"], rb["out"])


def test_bf16_state_variant_is_the_rounded_float_step():
    # three tokens of the bf16-state variant == three plain steps with the state
    # and the outputs rounded to bf16 after each step (by the pinned rounding)
    shape, inp = _small(B=2, T=3, Hq=1, Hv=2)
    rnd = np.vectorize(oracle.round_bf16)
    st0 = rnd(inp["state"]).astype(np.float32)                # a bf16 starting state
    lp = oracle.layer(inp["x"], inp["z"], inp["alpha"], inp["beta_logit"], inp["conv_w"],
                      inp["dt"], inp["A_log"], inp["norm_w"], st0, inp["hist"], Hq=shape.Hq,
                      W=shape.W, bf16_state=True)
    st, hi = st0, inp["hist"]
    for t in range(shape.T):
        one = oracle.layer(inp["x"][:, t:t + 1], inp["z"][:, t:t + 1], inp["alpha"][:, t:t + 1],
                           inp["beta_logit"][:, t:t + 1], inp["conv_w"], inp["dt"], inp["A_log"],
                           inp["norm_w"], st, hi, Hq=shape.Hq, W=shape.W)
        np.testing.assert_array_equal(lp["out"][:, t], rnd(one["out"][:, 0]))
        st = rnd(one["state"])          # exact in float32: bf16 values
        assert np.array_equal(st.astype(np.float32).astype(np.float64), st)
        st = st.astype(np.float32)
        hi = one["hist"]
    np.testing.assert_array_equal(lp["state"], st)
    np.testing.assert_array_equal(lp["hist"], hi)
