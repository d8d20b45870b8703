"""Pins for the fp64 oracle: each part checked against something other than itself.

Closed forms, library routines (numpy / scipy / exact rational arithmetic),
the explicit matrix form of the update, invariants, and the independent
chunked form. CPU only.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle
from oracle.chunked import chunked_scan

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------ scalar functions
def test_softplus_matches_logaddexp_below_guard():
    # Below the guard, the guarded softplus is log(1 + e^v): numpy's logaddexp(0, v).
    for v in np.concatenate([np.linspace(-30, 20, 501), [20.0]]):
        assert oracle.softplus(v) == pytest.approx(np.logaddexp(0.0, v), rel=1e-14, abs=1e-300)


def test_softplus_guard_is_identity_above_20_and_continuous():
    # "guarded at 20": strictly above 20 it returns v itself.
    for v in [20.0 + 1e-12, 20.5, 33.0, 1e4, 1e30]:
        assert oracle.softplus(v) == v
    # The jump at the guard is log1p(e^20) - 20 = log1p(e^-20) ~ 2.06e-9.
    jump = oracle.softplus(20.0) - 20.0
    assert jump == pytest.approx(math.exp(-20.0), rel=1e-6)
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)


def test_sigmoid_and_silu_match_scipy():
    for v in np.linspace(-40, 40, 321):
        assert oracle.sigmoid(v) == pytest.approx(expit(v), rel=1e-14, abs=1e-300)
        assert oracle.silu(v) == pytest.approx(v * expit(v), rel=1e-14, abs=1e-300)


def test_decay_gate_closed_forms():
    dt = np.array([0.0, 0.0, 0.5, -0.25], np.float32)
    A_log = np.array([0.0, math.log(4.0), 0.0, 1.0], np.float32)
    alpha = np.array([[0.0, 30.0, -0.5, 0.25]], np.float32)
    g = oracle.decay_gate(alpha, dt, A_log)[0]
    assert g[0] == pytest.approx(-math.log(2.0), rel=1e-15)       # a = -1, softplus(0) = ln 2
    assert g[1] == pytest.approx(-4.0 * 30.0, rel=1e-7)          # guard: softplus(30) = 30, a = -4
    assert g[2] == pytest.approx(-math.log(2.0), rel=1e-15)      # alpha + dt = 0
    a3 = -math.exp(float(np.float32(1.0)))
    assert g[3] == pytest.approx(a3 * np.logaddexp(0.0, 0.0), rel=1e-15)


def test_decay_gate_random_against_library_softplus():
    H, rows = 48, 64
    dt = RNG.uniform(-1, 1, H).astype(np.float32)
    A_log = RNG.uniform(0, math.log(16), H).astype(np.float32)
    alpha = RNG.standard_normal((rows, H)).astype(np.float32) * 8
    g = oracle.decay_gate(alpha, dt, A_log)
    v = alpha.astype(np.float64) + dt.astype(np.float64)
    sp = np.where(v > 20, v, np.logaddexp(0.0, v))
    np.testing.assert_allclose(g, -np.exp(A_log.astype(np.float64)) * sp, rtol=1e-14)
    assert np.all(g < 0) and np.all(np.exp(g) < 1) and np.all(np.exp(g) >= 0)


# ------------------------------------------------------------ conv + SiLU
def _conv_scan(x, w, hist):
    outs = []
    h = hist
    for t in range(x.shape[0]):
        o, h = oracle.conv_step(x[t], w, h)
        outs.append(o)
    return np.array(outs), h


@pytest.mark.parametrize("W", [2, 4, 8])
def test_conv_delta_kernels(W):
    C, T = 6, 11
    x = RNG.standard_normal((T, C)).astype(np.float32)
    hist = RNG.standard_normal((C, W - 1))
    # tap W-1 only: the current token passes through SiLU unchanged
    w = np.zeros((C, W), np.float32)
    w[:, W - 1] = 1
    out, _ = _conv_scan(x, w, hist)
    np.testing.assert_allclose(out, x * expit(x.astype(np.float64)), rtol=1e-15)
    # tap 0 only: the input delayed by W-1 tokens (from the history first)
    w = np.zeros((C, W), np.float32)
    w[:, 0] = 1
    out, hend = _conv_scan(x, w, hist)
    stream = np.concatenate([hist.T, x.astype(np.float64)], 0)     # [W-1+T][C], oldest first
    delayed = stream[:T]
    np.testing.assert_allclose(out, delayed * expit(delayed), rtol=1e-15)
    # the history ends holding the last W-1 RAW inputs
    np.testing.assert_array_equal(hend, stream[-(W - 1):].T)


def test_conv_general_taps_match_numpy_correlate():
    C, T, W = 5, 9, 4
    x = RNG.standard_normal((T, C)).astype(np.float32)
    w = (RNG.standard_normal((C, W)) * 0.5).astype(np.float32)
    hist = RNG.standard_normal((C, W - 1))
    out, _ = _conv_scan(x, w, hist)
    for c in range(C):
        stream = np.concatenate([hist[c], x[:, c].astype(np.float64)])
        pre = np.correlate(stream, w[c].astype(np.float64), mode="valid")
        np.testing.assert_allclose(out[:, c], pre * expit(pre), rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------ L2 norm
def test_l2norm_unit_norm_and_direction():
    v = RNG.standard_normal(128)
    u = oracle.l2norm(v, 0.0)
    assert np.linalg.norm(u) == pytest.approx(1.0, abs=1e-15)
    assert np.dot(u, v) / np.linalg.norm(v) == pytest.approx(1.0, abs=1e-14)
    # with eps, |u|^2 = s / (s + eps): a tiny vector stays well below unit length
    small = v * 1e-4
    s = float(np.dot(small, small))
    us = oracle.l2norm(small, 1e-6)
    assert np.dot(us, us) == pytest.approx(s / (s + 1e-6), rel=1e-13)
    assert np.dot(us, us) < 0.7


# ------------------------------------------------------------ recurrence
def test_recurrence_full_forget_gives_outer_product():
    # A_log = 10 and alpha + dt = 0: g = -e^10 ln 2 ~ -15267, exp(g) underflows to 0.
    g = oracle.decay_gate(np.zeros((1, 1), np.float32), np.zeros(1, np.float32),
                          np.full(1, 10.0, np.float32))[0, 0]
    assert math.exp(g) == 0.0
    d = 16
    S = RNG.standard_normal((d, d))
    q, k, v = RNG.standard_normal((3, d))
    S1, o = oracle.recurrence_step(S, q, k, v, g, 1.0, 1 / math.sqrt(d))
    np.testing.assert_array_equal(S1, np.outer(k, v))
    np.testing.assert_allclose(o, np.dot(q, k) * v / math.sqrt(d), rtol=1e-13, atol=1e-15)


def test_delta_rule_reads_back_written_value():
    # beta = 1, |k| = 1: after the write, S'^T k = v for any decay and prior state.
    d = 32
    for g in (-0.01, -1.0, -7.5):
        S = RNG.standard_normal((d, d))
        k = RNG.standard_normal(d)
        k /= np.linalg.norm(k)
        v = RNG.standard_normal(d)
        S1, _ = oracle.recurrence_step(S, k, k, v, g, 1.0, 1.0)
        np.testing.assert_allclose(S1.T @ k, v, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("d", [1, 2, 3])
def test_recurrence_matches_matrix_form(d):
    # "GDN staleness" (scr_state.hpp): S' = e^g (I - b k k^T) S + b k v^T.
    for _ in range(20):
        S = RNG.standard_normal((d, d))
        q, k, v = RNG.standard_normal((3, d))
        g = -abs(RNG.standard_normal()) * 3
        b = RNG.uniform(0.01, 0.99)
        scale = 1 / math.sqrt(d)
        S1, o = oracle.recurrence_step(S, q, k, v, g, b, scale)
        ref = math.exp(g) * (np.eye(d) - b * np.outer(k, k)) @ S + b * np.outer(k, v)
        np.testing.assert_allclose(S1, ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(o, scale * ref.T @ q, rtol=1e-12, atol=1e-13)


def test_recurrence_exact_rational_d2():
    # Exact arithmetic on a 2x2 example: decay 1/2 (g = -ln 2), beta 1/4.
    F = Fraction
    S = [[F(1), F(-2)], [F(3), F(1, 2)]]
    k = [F(1, 2), F(-1, 4)]
    v = [F(2), F(-1)]
    q = [F(-1), F(3, 2)]
    dec, b = F(1, 2), F(1, 4)
    Sd = [[dec * S[i][j] for j in range(2)] for i in range(2)]
    pred = [sum(Sd[i][j] * k[i] for i in range(2)) for j in range(2)]
    u = [b * (v[j] - pred[j]) for j in range(2)]
    S1 = [[Sd[i][j] + k[i] * u[j] for j in range(2)] for i in range(2)]
    o = [sum(S1[i][j] * q[i] for i in range(2)) for j in range(2)]
    fl = lambda m: np.array(m, dtype=np.float64)
    Sg, og = oracle.recurrence_step(fl(S), fl(q), fl(k), fl(v), -math.log(2.0), 0.25, 1.0)
    np.testing.assert_allclose(Sg, fl(S1), rtol=1e-15)
    np.testing.assert_allclose(og, fl(o), rtol=1e-15)


def test_contraction_bound():
    # |D_end|_F <= exp(sum_t g_t) |D_0|_F for |k| <= 1 and beta in (0, 1).
    d, T = 24, 12
    S1 = RNG.standard_normal((d, d))
    S2 = RNG.standard_normal((d, d))
    D0 = np.linalg.norm(S1 - S2)
    gsum = 0.0
    for _ in range(T):
        k = RNG.standard_normal(d)
        k /= np.linalg.norm(k) * RNG.uniform(1.0, 2.0)
        q, v = RNG.standard_normal((2, d))
        g = -RNG.uniform(0.0, 0.3)
        b = RNG.uniform(0.05, 0.95)
        S1, _ = oracle.recurrence_step(S1, q, k, v, g, b, 1.0)
        S2, _ = oracle.recurrence_step(S2, q, k, v, g, b, 1.0)
        gsum += g
    assert np.linalg.norm(S1 - S2) <= math.exp(gsum) * D0 * (1 + 1e-12)


def _prepared_inputs(T, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    a = -np.exp(rng.uniform(0, math.log(16)))
    g = a * np.logaddexp(0, rng.standard_normal(T) + rng.uniform(-1, 1))
    beta = expit(rng.standard_normal(T))
    S0 = rng.standard_normal((d, d)) * 0.1
    return q, k, v, g, beta, S0


@pytest.mark.parametrize("T,chunk", [(37, 1), (37, 4), (130, 16), (130, 64), (64, 64), (200, 64)])
def test_chunked_form_equals_sequential_scan(T, chunk):
    d = 32
    q, k, v, g, beta, S0 = _prepared_inputs(T, d, seed=T * 7 + chunk)
    scale = 1 / math.sqrt(d)
    S_seq, y_seq = oracle.recurrence_scan(q, k, v, g, beta, S0, scale)
    S_chk, y_chk = chunked_scan(q, k, v, g, beta, S0, chunk, scale)
    assert np.abs(S_chk - S_seq).max() <= 1e-12 * np.abs(S_seq).max()
    assert np.abs(y_chk - y_seq).max() <= 1e-12 * np.abs(y_seq).max()


def test_chunked_form_slow_decay():
    # weak decay keeps far-apart tokens coupled inside a chunk
    d, T = 16, 96
    q, k, v, _, beta, S0 = _prepared_inputs(T, d, seed=5)
    g = -np.full(T, 0.01)
    S_seq, y_seq = oracle.recurrence_scan(q, k, v, g, beta, S0, 0.25)
    S_chk, y_chk = chunked_scan(q, k, v, g, beta, S0, 64, 0.25)
    assert np.abs(S_chk - S_seq).max() <= 1e-11 * np.abs(S_seq).max()
    assert np.abs(y_chk - y_seq).max() <= 1e-11 * np.abs(y_seq).max()


# ------------------------------------------------------------ gated RMSNorm
def test_gated_norm_constant_head():
    d, eps = 128, 1e-6
    w = (1 + RNG.standard_normal(d) * 0.1).astype(np.float32)
    z = RNG.standard_normal(d)
    for c in (-3.0, 0.02, 5.0):
        out = oracle.gated_norm(np.full(d, c), w, z, eps)
        ref = np.sign(c) * w.astype(np.float64) * z * expit(z) / math.sqrt(1 + eps / c ** 2)
        np.testing.assert_allclose(out, ref, rtol=1e-14)
    assert np.all(oracle.gated_norm(RNG.standard_normal(d), w, np.zeros(d), eps) == 0)


def test_gated_norm_scale_invariant():
    d = 64
    w = np.ones(d, np.float32)
    y = RNG.standard_normal(d)
    z = RNG.standard_normal(d)
    a = oracle.gated_norm(y, w, z, 0.0)
    b = oracle.gated_norm(y * 37.5, w, z, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    # RMS of the normalised value (before the gate) is 1
    one = oracle.gated_norm(y, w, np.full(d, 50.0), 0.0) / (50.0 * expit(50.0))
    assert math.sqrt(np.mean(one ** 2)) == pytest.approx(1.0, rel=1e-13)


# ------------------------------------------------------------------ bf16 storage rounding
def test_round_bf16_closed_forms():
    r = oracle.round_bf16
    ulp1 = 2.0 ** -7                       # bf16 spacing in [1, 2)
    assert r(1.0) == 1.0 and r(-3.5) == -3.5 and r(0.0) == 0.0
    assert r(1.0 + ulp1 / 2) == 1.0                        # tie -> even (1.0)
    assert r(1.0 + 3 * ulp1 / 2) == 1.0 + 2 * ulp1          # tie -> even mantissa
    assert r(1.0 + ulp1 / 2 + 2.0 ** -40) == 1.0 + ulp1     # just above the tie: up
    assert r(1.0 + ulp1 / 2 - 2.0 ** -40) == 1.0            # just below: down
    assert r(-(1.0 + ulp1 / 2 + 2.0 ** -40)) == -(1.0 + ulp1)
    big = 2.0 ** 128 - 2.0 ** 120                          # largest finite bf16
    assert r(big) == big
    assert r(2.0 ** 128 - 2.0 ** 119) == math.inf          # tie above the largest: overflow
    assert r(2.0 ** 128 - 2.0 ** 119 - 2.0 ** 100) == big
    assert r(2.0 ** -133) == 2.0 ** -133                   # smallest subnormal
    assert r(2.0 ** -134) == 0.0                           # tie with zero -> zero
    assert r(3 * 2.0 ** -134) == 2.0 ** -132               # tie -> even
    assert math.isnan(r(math.nan)) and r(-math.inf) == -math.inf


def test_round_bf16_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    # for float32-representable inputs a single float32 -> bf16 RNE (torch's
    # conversion) is the same rounding; the draws include exact ties
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))).astype(np.float32)
    bits = x.view(np.uint32)
    ties = ((bits & ~np.uint32(0xFFFF)) | np.uint32(0x8000)).view(np.float32)[:500]
    vals = np.concatenate([x, ties])
    want = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    np.testing.assert_array_equal(got, want)
