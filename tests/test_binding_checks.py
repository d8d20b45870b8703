"""The Python binding refuses tensors it cannot hand to a kernel, before the library call.

A host tensor's address given to a kernel faults the GPU; a tensor of another
dtype or layout than the call reads gives wrong results silently. The checks
run in the order dtype, layout, device, so all three are reachable with host
tensors here (no GPU needed). Raw integer addresses stay unchecked: the ABI
tests use them on purpose.
"""
import pytest

torch = pytest.importorskip("torch")

import gated_delta_ssm_gb300 as gdn  # noqa: E402

FAKE = 1 << 20                     # an address that is never dereferenced: every call raises first
PRM = gdn.Params(FAKE, FAKE, FAKE, FAKE)
DIMS = gdn.Dims(n_seq=2, n_qk_heads=1, n_v_heads=1)     # conv_dim 384, rows of x 384 apart


def _state(**kw):
    return torch.zeros(2, 1, 128, 128, **kw)


def test_state_of_another_dtype_is_refused():
    with pytest.raises(TypeError, match="state: dtype torch.float64"):
        gdn.decode_step(_state(dtype=torch.float64), FAKE, FAKE, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)
    with pytest.raises(TypeError, match="state: dtype torch.float32, expected bfloat16"):
        gdn.decode_step_bf16_state(_state(), FAKE, FAKE, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)


def test_non_contiguous_state_is_refused():
    st = _state().transpose(2, 3)
    with pytest.raises(ValueError, match="state: tensor must be contiguous"):
        gdn.decode_step(st, FAKE, FAKE, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)


def test_host_tensor_is_refused():
    with pytest.raises(ValueError, match="not on a CUDA device"):
        gdn.decode_step(_state(), FAKE, FAKE, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)
    with pytest.raises(ValueError, match="params.conv_w: tensor is on cpu"):
        gdn.decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                        gdn.Params(torch.zeros(384, 4), FAKE, FAKE, FAKE), FAKE, DIMS)


def test_activation_rows_must_match_the_dims_strides():
    # x rows 384 elements apart: a [2][1][384] tensor, or a token slice of a longer buffer
    # whose stride the dims state
    ok = torch.zeros(2, 1, 384)
    with pytest.raises(ValueError, match="not on a CUDA device"):   # layout accepted
        gdn.decode_step(FAKE, FAKE, ok, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)
    wide = torch.zeros(2, 1, 512)[..., :384]                        # rows 512 apart
    with pytest.raises(ValueError, match="x: dimension 0 steps 512 elements"):
        gdn.decode_step(FAKE, FAKE, wide, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)
    strided = torch.zeros(2, 1, 768)[..., ::2]                      # elements 2 apart
    with pytest.raises(ValueError, match="x: elements of a row must be contiguous"):
        gdn.decode_step(FAKE, FAKE, strided, FAKE, FAKE, FAKE, PRM, FAKE, DIMS)
    buf = torch.zeros(2, 3, 384)                                    # token 1 of 3 per sequence
    d3 = gdn.Dims(n_seq=2, n_qk_heads=1, n_v_heads=1, x_stride=3 * 384, z_stride=3 * 128,
                  gate_stride=3)
    with pytest.raises(ValueError, match="not on a CUDA device"):
        gdn.decode_step(FAKE, FAKE, buf[:, 1], FAKE, FAKE, FAKE, PRM, FAKE, d3)
    with pytest.raises(ValueError, match="x: dimension 0 steps 1152 elements"):
        gdn.decode_step(FAKE, FAKE, buf[:, 1], FAKE, FAKE, FAKE, PRM, FAKE, DIMS)


def test_activations_share_one_dtype():
    x = torch.zeros(2, 1, 384, dtype=torch.bfloat16)
    z = torch.zeros(2, 1, 128)
    with pytest.raises(TypeError, match="z: dtype torch.float32, x is torch.bfloat16"):
        gdn.decode_step(FAKE, FAKE, x, z, FAKE, FAKE, PRM, FAKE, DIMS)
    with pytest.raises(TypeError, match="x: dtype torch.float16"):
        gdn.decode_step(FAKE, FAKE, x.half(), FAKE, FAKE, FAKE, PRM, FAKE, DIMS)


def test_accept_counts_and_workspace_are_checked():
    with pytest.raises(TypeError, match="n_accept: dtype torch.int64"):
        gdn.verify_commit(FAKE, FAKE, FAKE, FAKE, torch.ones(2, dtype=torch.int64), DIMS)
    ws = torch.zeros(64, 2, dtype=torch.uint8).t()
    with pytest.raises(ValueError, match="workspace: tensor must be contiguous"):
        gdn.prefill_chunked(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, PRM, FAKE, DIMS, 64, 64,
                            workspace=ws)


def test_scan_inputs_are_checked():
    q = torch.zeros(2, 4, 384)
    with pytest.raises(TypeError, match="state: dtype torch.bfloat16"):
        gdn.recurrence_scan(_state(dtype=torch.bfloat16), q, q, q, 384, FAKE, FAKE, FAKE, DIMS, 4,
                            0.1)
    with pytest.raises(ValueError, match="q: dimension 1 steps 384 elements, the row stride "
                                         "makes it 256"):
        gdn.recurrence_scan(FAKE, q, FAKE, FAKE, 256, FAKE, FAKE, FAKE, DIMS, 4, 0.1)
