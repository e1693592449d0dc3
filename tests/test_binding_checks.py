"""The Python binding rejects malformed tensors before anything reaches the C ABI (which gets
only addresses and trusts the sizes). CPU tensors are enough: shapes and types are checked
before the device, so every check here runs without a GPU and without loading the library."""

import pytest

torch = pytest.importorskip("torch")

import rope_cu_tile_gb300 as pk  # noqa: E402


def inputs(T=8, H=2, half=32, dtype=torch.bfloat16):
    qkv = torch.zeros((T, 3 * H * 64), dtype=dtype)
    cos = torch.zeros((T, half), dtype=dtype)
    cu = torch.tensor([0, T], dtype=torch.int32)
    return qkv, cos, cos.clone(), cu


def test_attend_shape_and_type_checks():
    qkv, cos, sin, cu = inputs()
    with pytest.raises(ValueError, match="qkv"):
        pk.attend(qkv[:, :-1], cos, sin, cu, 2, 0, 0.125)
    with pytest.raises(ValueError, match=r"\[P, 32\]"):
        pk.attend(qkv, cos[:, :16], sin[:, :16], cu, 2, 0, 0.125)
    with pytest.raises(TypeError, match="cos/sin"):
        pk.attend(qkv, cos.float(), sin, cu, 2, 0, 0.125)
    with pytest.raises(TypeError, match="cu"):
        pk.attend(qkv, cos, sin, cu.float(), 2, 0, 0.125)
    with pytest.raises(ValueError, match="CUDA"):
        pk.attend(qkv, cos, sin, cu, 2, 0, 0.125)


def test_backward_and_rope_checks():
    qkv, cos, sin, cu = inputs()
    out = torch.zeros((8, 128), dtype=torch.bfloat16)
    lse = torch.zeros((2, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="qkv"):
        pk.attend_backward(qkv[:, :-64], cos, sin, cu, 2, 0, 0.125, out, lse, out)
    with pytest.raises(ValueError, match="CUDA"):
        pk.attend_backward(qkv, cos, sin, cu, 2, 0, 0.125, out, lse, out)
    with pytest.raises(ValueError, match=r"\[P, 16\]"):
        pk.rope(qkv, cos, sin, cu, 2, dims=32)
    q32, c16, s16, cu32 = inputs(half=16)
    with pytest.raises(ValueError, match="CUDA"):
        pk.rope(q32, c16, s16, cu32, 2, dims=32)


def test_buffer_check():
    t = torch.zeros((4, 64), dtype=torch.float16)
    with pytest.raises(ValueError, match="out must be"):
        pk._need(t, (4, 128), torch.float16, "out")
    with pytest.raises(ValueError, match="out must be"):
        pk._need(t, (4, 64), torch.bfloat16, "out")
    with pytest.raises(ValueError, match="contiguous CUDA"):
        pk._need(t, (4, 64), torch.float16, "out")  # right shape and type, but on the host
