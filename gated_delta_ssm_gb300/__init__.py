"""gated_delta_ssm_gb300 -- Python binding of libgdn, the gated-delta SSM layer step on GB300.

Argument marshalling only: every entry point forwards device pointers, sizes
and the current CUDA stream to the function of the same name in libgdn.so
(declared in include/gdn.h) and raises on a non-OK status. There is no
fallback: if the compiled library is missing or fails to load, every call
raises.

Tensors are torch CUDA tensors (PyTorch supplies device memory and streams);
activations may be float32 or bfloat16, everything else is float32.
"""
from __future__ import annotations

import ctypes as _ct
import dataclasses as _dc
import os as _os
import threading as _th

__all__ = [
    "Dims", "Params", "GdnError", "load", "library_path",
    "decay_gate", "conv_update", "recurrence_decode", "gated_norm",
    "decode_step", "decode_step_select", "verify_k2", "verify_commit", "prefill_chunked",
    "prefill_workspace_bytes",
    "recurrence_scan",
    "layer_scan", "verify_kn", "verify_commit_kn", "decode_step_bf16_state", "check_device",
    "version",
]

_PKG = _os.path.dirname(_os.path.abspath(__file__))
# GDN_CHECKED=1 selects the checked build (index range checks reported as device error
# bit 32; see gdn_check_device)
_LIB_PATH = _os.path.join(_PKG, "libgdn_checked.so" if _os.environ.get("GDN_CHECKED") == "1"
                          else "libgdn.so")
_lib = None
_lock = _th.Lock()

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE = 0, 1, 2, 3, 4
GDN_F32, GDN_BF16 = 0, 1


class GdnError(RuntimeError):
    def __init__(self, status: int, fn: str, detail: str = ""):
        self.status = status
        names = {1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_CUDA",
                 4: "GDN_ERR_DEVICE"}
        super().__init__(f"{fn}: {names.get(status, status)}" + (f" ({detail})" if detail else ""))


class _CDims(_ct.Structure):
    _fields_ = [("n_seq", _ct.c_int32), ("n_qk_heads", _ct.c_int32), ("n_v_heads", _ct.c_int32),
                ("head_dim", _ct.c_int32), ("d_conv", _ct.c_int32), ("reserved", _ct.c_int32),
                ("x_stride", _ct.c_int64), ("z_stride", _ct.c_int64), ("gate_stride", _ct.c_int64)]


class _CParams(_ct.Structure):
    _fields_ = [("conv_w", _ct.c_void_p), ("dt", _ct.c_void_p), ("A_log", _ct.c_void_p),
                ("norm_w", _ct.c_void_p), ("l2_eps", _ct.c_float), ("rms_eps", _ct.c_float)]


@_dc.dataclass
class Dims:
    """Shape of a layer call (see gdn_dims in include/gdn.h). Strides are in elements."""
    n_seq: int
    n_qk_heads: int
    n_v_heads: int
    head_dim: int = 128
    d_conv: int = 4
    x_stride: int = 0       # 0 -> conv_dim
    z_stride: int = 0       # 0 -> n_v_heads * head_dim
    gate_stride: int = 0    # 0 -> n_v_heads

    @property
    def conv_dim(self) -> int:
        return (2 * self.n_qk_heads + self.n_v_heads) * self.head_dim

    def c(self) -> _CDims:
        return _CDims(self.n_seq, self.n_qk_heads, self.n_v_heads, self.head_dim, self.d_conv, 0,
                      self.x_stride or self.conv_dim, self.z_stride or self.n_v_heads * self.head_dim,
                      self.gate_stride or self.n_v_heads)


@_dc.dataclass
class Params:
    """Per-layer float32 parameters (device tensors)."""
    conv_w: object
    dt: object
    A_log: object
    norm_w: object
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6

    def c(self) -> _CParams:
        return _CParams(_dev(self.conv_w, "params.conv_w", _F32), _dev(self.dt, "params.dt", _F32),
                        _dev(self.A_log, "params.A_log", _F32),
                        _dev(self.norm_w, "params.norm_w", _F32), self.l2_eps, self.rms_eps)


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libgdn.so (built by __graft_entry__.build() or gated_delta_ssm_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _os.path.exists(_LIB_PATH):
            raise ImportError(f"libgdn.so is not built ({_LIB_PATH}); run "
                              "`python -m gated_delta_ssm_gb300.build`")
        L = _ct.CDLL(_LIB_PATH)
        vp, i32, i64, f32 = _ct.c_void_p, _ct.c_int32, _ct.c_int64, _ct.c_float
        pd, pp = _ct.POINTER(_CDims), _ct.POINTER(_CParams)
        sigs = {
            "gdn_decay_gate": [vp, _ct.c_int, i64, vp, vp, vp, i32, i32, vp],
            "gdn_conv_update": [vp, vp, _ct.c_int, vp, vp, pd, i32, f32, vp],
            "gdn_recurrence_decode": [vp, vp, vp, vp, i64, vp, vp, vp, pd, f32, vp],
            "gdn_gated_norm": [vp, vp, vp, _ct.c_int, i64, vp, i32, i32, i32, f32, vp],
            "gdn_decode_step": [vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, vp],
            "gdn_decode_step_bf16_state": [vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, vp],
            "gdn_verify_k2": [vp, vp, vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, vp],
            "gdn_decode_step_select": [vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, vp, _ct.c_int, pp,
                                       vp, pd, vp],
            "gdn_verify_commit": [vp, vp, vp, vp, vp, pd, vp],
            "gdn_prefill_chunked": [vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, i32, i32, vp,
                                    _ct.c_size_t, vp],
            "gdn_recurrence_scan": [vp, vp, vp, vp, i64, vp, vp, vp, pd, i32, f32, vp],
            "gdn_layer_scan": [vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, i32, vp],
            "gdn_verify_kn": [vp, vp, vp, vp, vp, vp, vp, vp, _ct.c_int, pp, vp, pd, i32, vp],
            "gdn_verify_commit_kn": [vp, vp, vp, vp, vp, pd, i32, vp],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _ct.c_int
        for name in ("gdn_last_cuda_error", "gdn_version"):
            getattr(L, name).restype = _ct.c_char_p
            getattr(L, name).argtypes = []
        L.gdn_prefill_workspace_bytes.restype = _ct.c_size_t
        L.gdn_prefill_workspace_bytes.argtypes = [pd, i32, i32]
        L.gdn_testing_set_first_wait_ns.restype = None
        L.gdn_testing_set_first_wait_ns.argtypes = [_ct.c_uint64]
        L.gdn_testing_row_splits.restype = None
        L.gdn_testing_row_splits.argtypes = [i32, i32, i32, i32, _ct.POINTER(_ct.c_int32),
                                             _ct.POINTER(_ct.c_int32)]
        L.gdn_check_device.restype = _ct.c_int
        L.gdn_check_device.argtypes = [_ct.POINTER(_ct.c_int32)]
        L.gdn_status_string.restype = _ct.c_char_p
        L.gdn_status_string.argtypes = [_ct.c_int]
        _lib = L
    return _lib


def check_device() -> int:
    """Synchronise, then read and clear the device-side error word (0 = no kernel gave up a wait)."""
    code = _ct.c_int32(0)
    st = load().gdn_check_device(_ct.byref(code))
    if st not in (GDN_OK, GDN_ERR_DEVICE):
        _check(st, "gdn_check_device")
    return int(code.value)


def version() -> str:
    return load().gdn_version().decode()


# ------------------------------------------------------------------ marshalling helpers
def _torch_dtypes(*names):
    import torch
    return tuple(getattr(torch, n) for n in names)


_F32, _ACT, _I32 = ("float32",), ("float32", "bfloat16"), ("int32",)


def _dev(t, name: str, dtypes=None, row_stride: int | None = None) -> int | None:
    """Device address of a tensor argument, once it is known to be safe to hand to a kernel:
    of one of `dtypes` (torch dtype names), laid out as the call reads it (contiguous, or, when
    row_stride is given, elements contiguous within a row and every leading index a whole
    number of rows of row_stride elements), and a CUDA tensor on the current device. None
    stays None; an int is taken as a raw device address, unchecked."""
    if t is None or isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor, got {type(t).__name__}")
    if dtypes is not None and t.dtype not in _torch_dtypes(*dtypes):
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(dtypes)}")
    if row_stride is None:
        if not t.is_contiguous():
            raise ValueError(f"{name}: tensor must be contiguous")
    elif t.numel() > 0:
        if t.dim() == 0 or t.stride(-1) != 1:
            raise ValueError(f"{name}: elements of a row must be contiguous")
        expected = row_stride
        for d in range(t.dim() - 2, -1, -1):
            if t.size(d) > 1 and t.stride(d) != expected:
                raise ValueError(f"{name}: dimension {d} steps {t.stride(d)} elements, the "
                                 f"row stride makes it {expected}")
            expected *= t.size(d)
    if not t.is_cuda:
        raise ValueError(f"{name}: tensor is on {t.device}, not on a CUDA device")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: tensor is on {t.device}, the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    return t.data_ptr()


def _ptr(t) -> int | None:
    """Address of an untyped buffer (a workspace): contiguous, CUDA, current device."""
    return _dev(t, "workspace")


def _acts(x, z, alpha, beta_logit, cd) -> tuple:
    """The activation inputs of a layer call: one dtype (float32 or bfloat16) for all four,
    rows of x, z and the gates at the strides of dims."""
    if x is not None and not isinstance(x, int):
        for t, nm in ((z, "z"), (alpha, "alpha"), (beta_logit, "beta_logit")):
            if t is not None and not isinstance(t, int) and t.dtype != x.dtype:
                raise TypeError(f"{nm}: dtype {t.dtype}, x is {x.dtype}")
    return (_dev(x, "x", _ACT, cd.x_stride), _dev(z, "z", _ACT, cd.z_stride),
            _dev(alpha, "alpha", _ACT, cd.gate_stride),
            _dev(beta_logit, "beta_logit", _ACT, cd.gate_stride))


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"activation dtype must be float32 or bfloat16, got {t.dtype}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, fn: str):
    if status != GDN_OK:
        detail = load().gdn_last_cuda_error().decode() if status == GDN_ERR_CUDA else ""
        raise GdnError(status, fn, detail)


# ------------------------------------------------------------------ entry points
def decay_gate(alpha, dt, A_log, g, rows: int, n_heads: int, alpha_stride: int = 0, stream=None):
    _check(load().gdn_decay_gate(_dev(alpha, "alpha", _ACT, alpha_stride or n_heads), _dtype(alpha),
                                 alpha_stride or n_heads, _dev(dt, "dt", _F32),
                                 _dev(A_log, "A_log", _F32), _dev(g, "g", _F32), rows, n_heads,
                                 _stream(stream)),
           "gdn_decay_gate")


def conv_update(conv_state, x, conv_w, out, dims: Dims, n_tokens: int = 1, l2_eps: float = 1e-6,
                stream=None):
    cd = dims.c()
    _check(load().gdn_conv_update(_dev(conv_state, "conv_state", _F32),
                                  _dev(x, "x", _ACT, cd.x_stride), _dtype(x),
                                  _dev(conv_w, "conv_w", _F32), _dev(out, "out", _F32),
                                  _ct.byref(cd), n_tokens, l2_eps, _stream(stream)),
           "gdn_conv_update")


def recurrence_decode(state, q, k, v, qkv_stride: int, g, beta, y, dims: Dims, scale: float,
                      stream=None):
    cd = dims.c()
    _check(load().gdn_recurrence_decode(_dev(state, "state", _F32),
                                        _dev(q, "q", _F32, qkv_stride), _dev(k, "k", _F32, qkv_stride),
                                        _dev(v, "v", _F32, qkv_stride), qkv_stride,
                                        _dev(g, "g", _F32), _dev(beta, "beta", _F32),
                                        _dev(y, "y", _F32), _ct.byref(cd), scale, _stream(stream)),
           "gdn_recurrence_decode")


def gated_norm(y, norm_w, z, out, rows: int, n_v_heads: int, head_dim: int = 128,
               z_stride: int = 0, eps: float = 1e-6, stream=None):
    zs = z_stride or n_v_heads * head_dim
    _check(load().gdn_gated_norm(_dev(y, "y", _F32), _dev(norm_w, "norm_w", _F32),
                                 _dev(z, "z", _ACT, zs), _dtype(z), zs, _dev(out, "out", _F32),
                                 rows, n_v_heads, head_dim, eps, _stream(stream)),
           "gdn_gated_norm")


def decode_step(state, conv_state, x, z, alpha, beta_logit, params: Params, out, dims: Dims,
                stream=None):
    cd, cp = dims.c(), params.c()
    _check(load().gdn_decode_step(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                  *_acts(x, z, alpha, beta_logit, cd), _dtype(x), _ct.byref(cp),
                                  _dev(out, "out", _F32), _ct.byref(cd), _stream(stream)),
           "gdn_decode_step")


def decode_step_bf16_state(state, conv_state, x, z, alpha, beta_logit, params: Params, out,
                           dims: Dims, stream=None):
    """state and out are bfloat16 tensors; see gdn_decode_step_bf16_state."""
    cd, cp = dims.c(), params.c()
    _check(load().gdn_decode_step_bf16_state(_dev(state, "state", ("bfloat16",)),
                                             _dev(conv_state, "conv_state", _F32),
                                             *_acts(x, z, alpha, beta_logit, cd), _dtype(x),
                                             _ct.byref(cp), _dev(out, "out", ("bfloat16",)),
                                             _ct.byref(cd), _stream(stream)),
           "gdn_decode_step_bf16_state")


def decode_step_select(state, conv_state, state_snap, conv_snap, conv_snap_entries: int, n_accept,
                       n_draft: int, x, z, alpha, beta_logit, params: Params, out, dims: Dims,
                       stream=None):
    """The step after a K-token verify, each sequence starting from the snapshot its accepted
    count selects; see gdn_decode_step_select."""
    cd, cp = dims.c(), params.c()
    _check(load().gdn_decode_step_select(_dev(state, "state", _F32),
                                         _dev(conv_state, "conv_state", _F32),
                                         _dev(state_snap, "state_snap", _F32),
                                         _dev(conv_snap, "conv_snap", _F32), conv_snap_entries,
                                         _dev(n_accept, "n_accept", _I32), n_draft,
                                         *_acts(x, z, alpha, beta_logit, cd), _dtype(x),
                                         _ct.byref(cp), _dev(out, "out", _F32), _ct.byref(cd),
                                         _stream(stream)),
           "gdn_decode_step_select")


def verify_k2(state, conv_state, state_snap, conv_snap, x, z, alpha, beta_logit, params: Params,
              out, dims: Dims, stream=None):
    cd, cp = dims.c(), params.c()
    _check(load().gdn_verify_k2(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                _dev(state_snap, "state_snap", _F32),
                                _dev(conv_snap, "conv_snap", _F32),
                                *_acts(x, z, alpha, beta_logit, cd), _dtype(x), _ct.byref(cp),
                                _dev(out, "out", _F32), _ct.byref(cd), _stream(stream)),
           "gdn_verify_k2")


def verify_commit(state, conv_state, state_snap, conv_snap, n_accept, dims: Dims, stream=None):
    cd = dims.c()
    _check(load().gdn_verify_commit(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                    _dev(state_snap, "state_snap", _F32),
                                    _dev(conv_snap, "conv_snap", _F32),
                                    _dev(n_accept, "n_accept", _I32), _ct.byref(cd),
                                    _stream(stream)),
           "gdn_verify_commit")


def prefill_workspace_bytes(dims: Dims, n_tokens: int, chunk: int = 64) -> int:
    """Bytes of device workspace gdn_prefill_chunked needs (0 for invalid arguments)."""
    cd = dims.c()
    return int(load().gdn_prefill_workspace_bytes(_ct.byref(cd), n_tokens, chunk))


def prefill_chunked(state, conv_state, x, z, alpha, beta_logit, params: Params, out, dims: Dims,
                    n_tokens: int, chunk: int = 64, workspace=None, stream=None):
    """workspace: a device tensor of at least prefill_workspace_bytes(dims, n_tokens, chunk)
    bytes; when None, one is allocated with torch for this call."""
    cd, cp = dims.c(), params.c()
    if workspace is None:
        import torch
        nbytes = prefill_workspace_bytes(dims, n_tokens, chunk)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    ws = _ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().gdn_prefill_chunked(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                      *_acts(x, z, alpha, beta_logit, cd), _dtype(x), _ct.byref(cp),
                                      _dev(out, "out", _F32), _ct.byref(cd), n_tokens, chunk, ws,
                                      ws_bytes, _stream(stream)),
           "gdn_prefill_chunked")


def testing_set_first_wait_ns(ns: int):
    """Test hook (include/gdn_testing.h): limit of the prefill's and the tiled conv's first
    bounded wait, in GPU global-timer nanoseconds, for later calls (0 = default)."""
    load().gdn_testing_set_first_wait_ns(int(ns))


def testing_row_splits(n_seq: int, n_v_heads: int, r: int, sms: int) -> tuple:
    """Test hook (include/gdn_testing.h): (decode, scan) row slices per V head the launchers
    choose on a device with `sms` SMs. Host-only."""
    d, s = _ct.c_int32(0), _ct.c_int32(0)
    load().gdn_testing_row_splits(n_seq, n_v_heads, r, sms, _ct.byref(d), _ct.byref(s))
    return d.value, s.value


def recurrence_scan(state, q, k, v, qkv_stride: int, g, beta, y, dims: Dims, n_tokens: int,
                    scale: float, stream=None):
    cd = dims.c()
    _check(load().gdn_recurrence_scan(_dev(state, "state", _F32),
                                      _dev(q, "q", _F32, qkv_stride), _dev(k, "k", _F32, qkv_stride),
                                      _dev(v, "v", _F32, qkv_stride), qkv_stride,
                                      _dev(g, "g", _F32), _dev(beta, "beta", _F32),
                                      _dev(y, "y", _F32), _ct.byref(cd), n_tokens, scale,
                                      _stream(stream)),
           "gdn_recurrence_scan")


def layer_scan(state, conv_state, x, z, alpha, beta_logit, params: Params, out, dims: Dims,
               n_tokens: int, stream=None):
    cd, cp = dims.c(), params.c()
    _check(load().gdn_layer_scan(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                 *_acts(x, z, alpha, beta_logit, cd), _dtype(x), _ct.byref(cp),
                                 _dev(out, "out", _F32), _ct.byref(cd), n_tokens,
                                 _stream(stream)),
           "gdn_layer_scan")


def verify_kn(state, conv_state, state_snap, conv_snap, x, z, alpha, beta_logit, params: Params,
              out, dims: Dims, n_draft: int, stream=None):
    cd, cp = dims.c(), params.c()
    _check(load().gdn_verify_kn(_dev(state, "state", _F32), _dev(conv_state, "conv_state", _F32),
                                _dev(state_snap, "state_snap", _F32),
                                _dev(conv_snap, "conv_snap", _F32),
                                *_acts(x, z, alpha, beta_logit, cd), _dtype(x), _ct.byref(cp),
                                _dev(out, "out", _F32), _ct.byref(cd), n_draft, _stream(stream)),
           "gdn_verify_kn")


def verify_commit_kn(state, conv_state, state_snap, conv_snap, n_accept, dims: Dims, n_draft: int,
                     stream=None):
    cd = dims.c()
    _check(load().gdn_verify_commit_kn(_dev(state, "state", _F32),
                                       _dev(conv_state, "conv_state", _F32),
                                       _dev(state_snap, "state_snap", _F32),
                                       _dev(conv_snap, "conv_snap", _F32),
                                       _dev(n_accept, "n_accept", _I32), _ct.byref(cd), n_draft,
                                       _stream(stream)),
           "gdn_verify_commit_kn")
