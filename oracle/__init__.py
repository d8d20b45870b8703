"""fp64 CPU oracle for the gated-delta SSM layer step (test infrastructure).

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package. The product path (the CUDA library and its
binding) never does, and this package imports nothing from it.

``gdn_oracle.c`` holds the arithmetic (plain C, double precision, one token
at a time); this module compiles it with gcc, loads it with ctypes, and
converts between numpy arrays and the C calls. The only transformation done
here is a layout change of the recurrent state between the library's
``[Hv][d_v][d_k]`` layout (row j contiguous over i) and the oracle's plain
``S[h][i][j]``. ``chunked.py`` holds an independent fp64 chunked form of the
recurrence that exists only to be compared against the sequential scan.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes as _ct
import os as _os
import subprocess as _sp
import threading as _th

import numpy as _np

_HERE = _os.path.dirname(_os.path.abspath(__file__))
_SRC = _os.path.join(_HERE, "gdn_oracle.c")
_LIB = _os.path.join(_HERE, "liboracle.so")
_lock = _th.Lock()
_lib = None

_D = _ct.POINTER(_ct.c_double)
_F = _ct.POINTER(_ct.c_float)


def build(force: bool = False) -> str:
    """Compile the C oracle into ``liboracle.so`` (gcc, no fast-math, no FMA contraction)."""
    if force or not _os.path.exists(_LIB) or _os.path.getmtime(_LIB) < _os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{_os.getpid()}"
        _sp.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                        "-shared", "-o", tmp, _SRC, "-lm"])
        _os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = _ct.CDLL(_LIB)
            L.gdnref_softplus.restype = _ct.c_double
            L.gdnref_softplus.argtypes = [_ct.c_double]
            L.gdnref_sigmoid.restype = _ct.c_double
            L.gdnref_sigmoid.argtypes = [_ct.c_double]
            L.gdnref_silu.restype = _ct.c_double
            L.gdnref_silu.argtypes = [_ct.c_double]
            L.gdnref_decay_gate.restype = None
            L.gdnref_decay_gate.argtypes = [_F, _F, _F, _D, _ct.c_long, _ct.c_int]
            L.gdnref_conv_step.restype = None
            L.gdnref_conv_step.argtypes = [_F, _F, _D, _D, _ct.c_int, _ct.c_int]
            L.gdnref_l2norm.restype = None
            L.gdnref_l2norm.argtypes = [_D, _ct.c_int, _ct.c_double]
            L.gdnref_recurrence_step.restype = None
            L.gdnref_recurrence_step.argtypes = [_D, _D, _D, _D, _ct.c_double, _ct.c_double,
                                                 _D, _ct.c_int, _ct.c_double]
            L.gdnref_gated_norm.restype = None
            L.gdnref_gated_norm.argtypes = [_D, _F, _D, _D, _ct.c_int, _ct.c_double]
            L.gdnref_layer.restype = _ct.c_int
            L.gdnref_layer.argtypes = [
                _ct.c_int, _ct.c_int, _ct.c_int, _ct.c_int, _ct.c_int,
                _F, _ct.c_long, _F, _ct.c_long, _F, _F,
                _F, _F, _F, _F, _ct.c_double, _ct.c_double,
                _D, _D, _D, _D, _D, _D, _D,
                _ct.c_int, _D, _D, _ct.c_int]
            L.gdnref_round_bf16.restype = _ct.c_double
            L.gdnref_round_bf16.argtypes = [_ct.c_double]
            L.gdnref_recurrence_scan.restype = None
            L.gdnref_recurrence_scan.argtypes = [_ct.c_int, _ct.c_int, _D, _D, _D, _D, _D,
                                                 _D, _D, _ct.c_double]
            _lib = L
    return _lib


def _f32(a):
    return _np.ascontiguousarray(a, dtype=_np.float32)


def _f64(a):
    return _np.ascontiguousarray(a, dtype=_np.float64)


def _pf(a):
    return a.ctypes.data_as(_F)


def _pd(a):
    return None if a is None else a.ctypes.data_as(_D)


# ---------------------------------------------------------------- scalar parts
def softplus(v: float) -> float:
    return lib().gdnref_softplus(float(v))


def sigmoid(v: float) -> float:
    return lib().gdnref_sigmoid(float(v))


def silu(v: float) -> float:
    return lib().gdnref_silu(float(v))


def decay_gate(alpha, dt, A_log):
    """g[rows][H] (pre-exp) from alpha[rows][H] and per-head dt, A_log."""
    alpha = _f32(alpha)
    rows, H = alpha.reshape(-1, alpha.shape[-1]).shape
    g = _np.empty((rows, H), _np.float64)
    lib().gdnref_decay_gate(_pf(alpha), _pf(_f32(dt)), _pf(_f32(A_log)), _pd(g), rows, H)
    return g.reshape(alpha.shape)


def conv_step(x, w, hist):
    """One conv+SiLU token. x [conv_dim], w [conv_dim][W], hist [conv_dim][W-1] (copied).
    Returns (out [conv_dim], new hist)."""
    x = _f32(x)
    w = _f32(w)
    h = _f64(hist).copy()
    cd, W = w.shape
    out = _np.empty(cd, _np.float64)
    lib().gdnref_conv_step(_pf(x), _pf(w), _pd(h), _pd(out), cd, W)
    return out, h


def l2norm(v, eps):
    v = _f64(v).copy()
    lib().gdnref_l2norm(_pd(v), v.size, float(eps))
    return v


def recurrence_step(S, q, k, v, g, beta, scale):
    """One head, plain orientation S[i][j] (copied). Returns (S', o)."""
    S = _f64(S).copy()
    d = S.shape[0]
    o = _np.empty(d, _np.float64)
    lib().gdnref_recurrence_step(_pd(S), _pd(_f64(q)), _pd(_f64(k)), _pd(_f64(v)),
                                 float(g), float(beta), _pd(o), d, float(scale))
    return S, o


def gated_norm(y, w, z, eps):
    y = _f64(y)
    out = _np.empty_like(y)
    lib().gdnref_gated_norm(_pd(y), _pf(_f32(w)), _pd(_f64(z)), _pd(out), y.size, float(eps))
    return out


def round_bf16(v: float) -> float:
    """Nearest bfloat16 value of a double, ties to even (gdnref_round_bf16)."""
    return lib().gdnref_round_bf16(float(v))


def recurrence_scan(q, k, v, g, beta, S, scale):
    """Sequential scan for one head: q,k,v [T][d], g, beta [T], S [d][d] plain (copied)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S = _f64(S).copy()
    T, d = q.shape
    y = _np.empty((T, d), _np.float64)
    lib().gdnref_recurrence_scan(T, d, _pd(q), _pd(k), _pd(v), _pd(g), _pd(beta),
                                 _pd(S), _pd(y), float(scale))
    return S, y


# ---------------------------------------------------------------- whole layer
def layer(x, z, alpha, beta_logit, conv_w, dt, A_log, norm_w, state_d1, hist,
          Hq, W, l2_eps=1e-6, rms_eps=1e-6, seqs=None, snap_after=-1,
          intermediates=False, threads=None, bf16_state=False, readout=False):
    """Run the layer over every token of each selected sequence.

    Activations are float32 arrays holding the exact input values
    (bf16 inputs already widened):
      x [B][T][>=conv_dim], z [B][T][>=Hv*d], alpha/beta_logit [B][T][Hv].
    state_d1 [B][Hv][d_v][d_k] and hist [B][conv_dim][W-1] are not modified.
    Returns a dict of float64 arrays for the selected sequences:
      out [b][T][Hv][d], state (library layout), hist, and with
      ``intermediates`` also conv [b][T][conv_dim], g, beta [b][T][Hv], y [b][T][Hv][d];
      with ``readout`` alone, y only (the readout before the gated norm);
      with snap_after >= 0 also state_snap, hist_snap.
    bf16_state runs the bf16-state variant: each head's state is rounded to
    bfloat16 after its step and each output value is rounded to bfloat16.
    Sequences run in parallel threads (the C call releases the GIL).
    """
    L = lib()
    B, T = x.shape[0], x.shape[1]
    Hv = alpha.shape[-1]
    d = norm_w.shape[0]
    cd = (2 * Hq + Hv) * d
    seqs = list(range(B)) if seqs is None else list(seqs)
    conv_w, dt, A_log, norm_w = map(_f32, (conv_w, dt, A_log, norm_w))
    nb = len(seqs)
    res = {"out": _np.empty((nb, T, Hv, d)), "state": _np.empty((nb, Hv, d, d)),
           "hist": _np.empty((nb, cd, W - 1))}
    if intermediates:
        res.update(conv=_np.empty((nb, T, cd)), g=_np.empty((nb, T, Hv)),
                   beta=_np.empty((nb, T, Hv)), y=_np.empty((nb, T, Hv, d)))
    elif readout:
        res.update(y=_np.empty((nb, T, Hv, d)))
    if snap_after >= 0:
        res.update(state_snap=_np.empty((nb, Hv, d, d)), hist_snap=_np.empty((nb, cd, W - 1)))

    def run(n):
        b = seqs[n]
        xb = _f32(x[b])
        zb = _f32(z[b])
        S = _f64(_np.swapaxes(state_d1[b], -1, -2))   # [h][i][j]
        hb = _f64(hist[b]).copy()
        out = _np.empty((T, Hv, d))
        inter = [None] * 4
        if intermediates:
            inter = [_np.empty((T, cd)), _np.empty((T, Hv)), _np.empty((T, Hv)),
                     _np.empty((T, Hv, d))]
        elif readout:
            inter[3] = _np.empty((T, Hv, d))
        Ss = hs = None
        if snap_after >= 0:
            Ss = _np.empty((Hv, d, d))
            hs = _np.empty((cd, W - 1))
        rc = L.gdnref_layer(T, Hq, Hv, d, W, _pf(xb), xb.shape[-1], _pf(zb), zb.shape[-1],
                            _pf(_f32(alpha[b])), _pf(_f32(beta_logit[b])),
                            _pf(conv_w), _pf(dt), _pf(A_log), _pf(norm_w),
                            float(l2_eps), float(rms_eps),
                            _pd(S), _pd(hb), _pd(out),
                            _pd(inter[0]), _pd(inter[1]), _pd(inter[2]), _pd(inter[3]),
                            int(snap_after), _pd(Ss), _pd(hs), int(bool(bf16_state)))
        if rc != 0:
            raise ValueError("oracle rejected the shape")
        res["out"][n] = out
        res["state"][n] = _np.swapaxes(S, -1, -2)
        res["hist"][n] = hb
        if intermediates:
            res["conv"][n], res["g"][n], res["beta"][n], res["y"][n] = inter
        elif readout:
            res["y"][n] = inter[3]
        if snap_after >= 0:
            res["state_snap"][n] = _np.swapaxes(Ss, -1, -2)
            res["hist_snap"][n] = hs

    nthreads = threads or min(nb, _os.cpu_count() or 1)
    if nthreads <= 1 or nb <= 1:
        for n in range(nb):
            run(n)
    else:
        with _cf.ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(run, range(nb)))
    return res
