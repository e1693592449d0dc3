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


class _FakeCuda:
    """Stands in for a contiguous CUDA tensor on a given device (no GPU needed): the checks
    read only shape, dtype, dim, device and contiguity before anything reaches the library."""

    def __init__(self, t, device):
        self._t = t
        self.device = torch.device(device)
        self.is_cuda = True
        self.shape = t.shape
        self.dtype = t.dtype

    def dim(self):
        return self._t.dim()

    def is_contiguous(self):
        return True


def test_tensors_on_different_devices_are_refused():
    qkv, cos, sin, cu = inputs()
    a = [_FakeCuda(x, "cuda:0") for x in (qkv, cos, sin, cu)]
    pk._check_inputs(*a, 2, 32)  # one device: accepted
    for k in range(1, 4):
        b = list(a)
        b[k] = _FakeCuda((qkv, cos, sin, cu)[k], "cuda:1")
        with pytest.raises(ValueError, match="different devices"):
            pk._check_inputs(*b, 2, 32)


def test_stream_of_another_device_is_refused():
    class S:
        device = torch.device("cuda:1")

    pk._check_stream(None, torch.device("cuda:0"))
    pk._check_stream(12345, torch.device("cuda:0"))  # a raw handle carries no device
    with pytest.raises(ValueError, match="stream"):
        pk._check_stream(S(), torch.device("cuda:0"))


def test_tables_shorter_than_a_sequence_are_refused():
    cu = torch.tensor([0, 5, 40, 41], dtype=torch.int32)
    pk._check_table_rows(cu, 35, 35)
    with pytest.raises(ValueError, match="positions"):
        pk._check_table_rows(cu, 34, 35)
    with pytest.raises(ValueError, match="positions"):
        pk._check_table_rows(cu, 34, None)  # the longest length read from cu: 35
