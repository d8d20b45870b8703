"""Shared helpers for the test suite: device upload, oracle runs, error metrics."""
from __future__ import annotations

import numpy as np

from gated_delta_ssm_gb300 import synth

OUT_TOL = 1e-3      # max relative error on layer outputs
STATE_TOL = 1e-4    # max relative error on the fp32 recurrent state
ELEM_FLOOR = 1e-3   # per-element metric: each element's error over max(|ref|, floor * row max)


def as_f32(a, dtype):
    """Exact float32 values of an activation array (bf16 bits or float32)."""
    if dtype == "bf16":
        return synth.bf16_to_f32(np.ascontiguousarray(a))
    return np.ascontiguousarray(a, np.float32)


def to_dev(a, dtype="f32"):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.cuda()


def device_inputs(shape: synth.Shape, inp: dict) -> dict:
    """Upload one workload; z stays a view into x when the shape keeps it in the row."""
    import torch
    dt = shape.act_dtype
    dev = {"x": to_dev(inp["x"], dt)}
    if shape.z_in_x:
        cd = shape.conv_dim
        dev["z"] = dev["x"][..., cd:cd + shape.Hv * shape.d]
    else:
        dev["z"] = to_dev(inp["z"], dt)
    for k in ("alpha", "beta_logit"):
        dev[k] = to_dev(inp[k], dt)
    for k in ("conv_w", "dt", "A_log", "norm_w", "state", "hist"):
        dev[k] = to_dev(inp[k])
    dev["accept"] = torch.from_numpy(inp["accept"]).cuda()
    return dev


def dims_of(shape: synth.Shape, rows_per_seq: int = 1):
    """ABI dims. rows_per_seq > 1 when single-token calls read one token slice
    ([:, t]) of a buffer that holds rows_per_seq tokens per sequence."""
    import gated_delta_ssm_gb300 as gdn
    m = rows_per_seq
    return gdn.Dims(n_seq=shape.B, n_qk_heads=shape.Hq, n_v_heads=shape.Hv, head_dim=shape.d,
                    d_conv=shape.W, x_stride=shape.xs * m,
                    z_stride=(shape.xs if shape.z_in_x else shape.Hv * shape.d) * m,
                    gate_stride=shape.Hv * m)


def params_of(dev: dict):
    import gated_delta_ssm_gb300 as gdn
    return gdn.Params(dev["conv_w"], dev["dt"], dev["A_log"], dev["norm_w"], 1e-6, 1e-6)


def run_oracle(shape: synth.Shape, inp: dict, T=None, seqs=None, **kw):
    import oracle
    T = shape.T if T is None else T
    dt = shape.act_dtype
    x = as_f32(inp["x"][:, :T], dt)
    z = as_f32(np.ascontiguousarray(inp["z"][:, :T]), dt)
    return oracle.layer(x, z, as_f32(inp["alpha"][:, :T], dt), as_f32(inp["beta_logit"][:, :T], dt),
                        inp["conv_w"], inp["dt"], inp["A_log"], inp["norm_w"], inp["state"],
                        inp["hist"], Hq=shape.Hq, W=shape.W, seqs=seqs, **kw)


def out_rel(x, ref):
    """Normwise relative error of layer outputs, one slice per (sequence, V head):
    max over slices of max|x - ref| / max|ref| over that head's tokens and
    channels. Outputs are [B][T][Hv][d] or [B][Hv][d] (one token)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if x.ndim == 3:
        x, ref = x[:, None], ref[:, None]
    num = np.abs(x - ref).max(axis=(1, 3))
    den = np.abs(ref).max(axis=(1, 3))
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def max_rel(x, ref, slice_axes: int):
    """Normwise relative error: max over slices (the trailing `slice_axes` axes form one
    slice) of max|x - ref| / max|ref| within the slice."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    lead = x.shape[:x.ndim - slice_axes]
    xf = x.reshape(int(np.prod(lead)) if lead else 1, -1)
    rf = ref.reshape(xf.shape)
    den = np.abs(rf).max(axis=1)
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(xf - rf).max(axis=1) / den).max())


def elem_rel(x, ref, floor=ELEM_FLOOR, y=None, rms_eps=1e-6):
    """Per-element relative error of layer outputs: each element's |x - ref| over
    max(|ref|, floor * max|ref| of its (sequence, V head) slice * gamma_row), the
    max over all elements. Outputs are [B][T][Hv][d] or [B][Hv][d] (one token).

    The floor is taken over the slice, not the token's own row: a token whose
    readout mean square m is far below rms_eps leaves the gated RMSNorm as a
    1/sqrt(rms_eps) scaling of its tiny readout, so its whole row is tiny.

    gamma_row (1 unless the reference readout y [.., Hv, d] is given) accounts
    for that conditioning: the norm multiplies a row's readout by its gain
    1/sqrt(m + rms_eps), so an absolute rounding error of the readout reaches the
    output gamma = gain_row / median gain of the slice times larger than on the
    slice's typical row (never less than 1)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if x.ndim == 3:
        x, ref = x[:, None], ref[:, None]
    slicemax = np.abs(ref).max(axis=(1, 3), keepdims=True)
    gamma = 1.0
    if y is not None:
        y = np.asarray(y, np.float64)
        if y.ndim == 3:
            y = y[:, None]
        gain = 1.0 / np.sqrt((y * y).mean(axis=-1, keepdims=True) + rms_eps)   # [B][T][Hv][1]
        gamma = np.maximum(1.0, gain / np.median(gain, axis=1, keepdims=True))
    den = np.maximum(np.abs(ref), floor * slicemax * gamma)
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(x - ref) / den).max())


def check_out(x, ref, tol=OUT_TOL, what="out", y=None):
    """Both output metrics within tol: normwise per (sequence, V head) and per element
    (with the reference readout y, the per-element floor follows the norm's gain)."""
    nr, er = out_rel(x, ref), elem_rel(x, ref, y=y)
    assert nr <= tol and er <= tol, f"{what}: normwise {nr:.3g}, per-element {er:.3g} (tol {tol:g})"
