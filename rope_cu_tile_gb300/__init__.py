"""Python binding of libpk: packed-sequence RoPE attention forward on GB300.

Argument marshalling only: every step of the computation runs in the CUDA library
(`libpk.so`, built from `csrc/` by `build.py`); there is no fallback of any kind. If the
library is missing or cannot load, every call raises.

The entry points mirror include/pk.h:
    attend(qkv, cos, sin, cu, H, window, scale, out=None, lse=None, stream=None, tuned=False)
    pk_attend(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)   (raw pointers)
    schedule(cu, T, window)      -> tile records [NT, 8]
    last_status(stream=None)     -> int
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpk.so")

PK_F32, PK_BF16, PK_F16 = 0, 1, 2
STATUS = {
    0: "PK_OK", 1: "PK_ERR_ARG", 2: "PK_ERR_ALIGN", 3: "PK_ERR_CUDA", 4: "PK_ERR_UNSUPPORTED",
    5: "PK_ERR_BAD_CU", 6: "PK_ERR_TIMEOUT", 7: "PK_ERR_NOMEM", 8: "PK_ERR_INTERNAL",
    9: "PK_ERR_TOO_LARGE", 10: "PK_ERR_CAPTURE",
}
NOALLOC_MAX_T = 1048576

# names declared in include/pk.h
EXPORTS = ("pk_attend", "pk_attend_bf16", "pk_attend_f16", "pk_attend_f32", "pk_attend_dt",
           "pk_schedule", "pk_schedule_capacity", "pk_last_status", "pk_status_string",
           "pk_version", "pk_release", "pk_profile_start", "pk_profile_stop", "pk_attend_noalloc", "pk_rope", "pk_attend_mixed",
           "pk_attend_backward", "pk_attend_tuned", "pk_tune_pick", "pk_tune_key", "pk_tune_clear",
           "pk_forward_kernel", "pk_kernel_name", "pk_attend_mixed_ops")
KERNELS = {0: "band", 1: "f32", 2: "tc", 3: "q4", 4: "tc_single", 5: "split"}

_lib = None


class PKError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = f"{STATUS.get(code, code)}: {status_string(code) if _lib else ''}"
        super().__init__(f"{what}: {msg}" if what else msg)


def load(path: str | None = None):
    """Load libpk.so (raises if it is missing: there is no other implementation)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpk.so not built ({p}); run __graft_entry__.build()")
    L = ctypes.CDLL(p)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    sig = [vp, vp, vp, vp, i32, i64, i32, i32, f32, vp, vp, vp]
    for name in ("pk_attend", "pk_attend_bf16", "pk_attend_f16", "pk_attend_f32"):
        getattr(L, name).argtypes = sig
        getattr(L, name).restype = i32
    L.pk_attend_dt.argtypes = [i32] + sig
    L.pk_attend_dt.restype = i32
    L.pk_attend_noalloc.argtypes = [i32] + sig[:11] + [vp, vp]
    L.pk_attend_noalloc.restype = i32
    L.pk_attend_backward.argtypes = [i32, vp, vp, vp, vp, i32, i64, i32, i32, f32, vp, vp, vp, vp, vp]
    L.pk_attend_backward.restype = i32
    L.pk_attend_mixed.argtypes = [i32] + sig
    L.pk_attend_mixed.restype = i32
    L.pk_attend_mixed_ops.argtypes = [i32] + sig
    L.pk_attend_mixed_ops.restype = i32
    L.pk_attend_tuned.argtypes = [i32, vp, vp, vp, vp, i32, i64, i32, i32, f32, i64, vp, vp, vp]
    L.pk_attend_tuned.restype = i32
    L.pk_tune_pick.argtypes = [i32, i32, i32, i64, i64]
    L.pk_tune_pick.restype = i32
    L.pk_tune_key.argtypes = [i32, i32, i32, i64, i64, ctypes.c_char_p, i32]
    L.pk_tune_key.restype = i32
    L.pk_tune_clear.argtypes = []
    L.pk_tune_clear.restype = i32
    L.pk_forward_kernel.argtypes = [i32, i32]
    L.pk_forward_kernel.restype = i32
    L.pk_kernel_name.argtypes = [i32]
    L.pk_kernel_name.restype = ctypes.c_char_p
    L.pk_rope.argtypes = [i32, vp, vp, vp, vp, i64, vp, i32, i64, i32, i32, i32, i32, vp, vp]
    L.pk_rope.restype = i32
    L.pk_schedule.argtypes = [vp, i32, i64, i32, vp, i64, ctypes.POINTER(i64), vp]
    L.pk_schedule.restype = i32
    L.pk_schedule_capacity.argtypes = [i64]
    L.pk_schedule_capacity.restype = i64
    L.pk_last_status.argtypes = [vp]
    L.pk_last_status.restype = i32
    L.pk_status_string.argtypes = [i32]
    L.pk_status_string.restype = ctypes.c_char_p
    L.pk_version.argtypes = []
    L.pk_version.restype = i32
    L.pk_release.argtypes = []
    L.pk_release.restype = i32
    L.pk_profile_start.argtypes = [i32]
    L.pk_profile_start.restype = i32
    dp = ctypes.POINTER(ctypes.c_double)
    L.pk_profile_stop.argtypes = [dp, dp, ctypes.POINTER(i32)]
    L.pk_profile_stop.restype = i32
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().pk_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise PKError(rc, what)


# ------------------------------------------------------------------------------------------
# raw-pointer entry points (same names and argument order as the C ABI)


def pk_attend(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream) -> int:
    return load().pk_attend(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)


def pk_attend_dt(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream) -> int:
    return load().pk_attend_dt(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)


def pk_attend_noalloc(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, status, stream) -> int:
    """The allocation-free variant (see include/pk.h): for callers that cannot let the library
    cudaMalloc a workspace; `status` is an optional device pointer to one int."""
    return load().pk_attend_noalloc(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, status, stream)


def pk_attend_mixed_ops(op_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream) -> int:
    """fp32 storage, 16-bit tensor-core operands, fp32 out (see include/pk.h)."""
    return load().pk_attend_mixed_ops(op_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)


def attend_mixed_ops(qkv, cos, sin, cu, H: int, window: int, scale: float, op_dtype, out=None, lse=None,
                     stream=None, max_len=None):
    """out [T, H*64] and lse [H, T], both float32, for float32 device tensors qkv [T, 3*H*64] and
    cos/sin [P, 32], the products on the tensor cores with operands of op_dtype
    (torch.float16 or torch.bfloat16)."""
    torch = _torch()
    if qkv.dtype != torch.float32:
        raise TypeError("qkv must be float32")
    _check_inputs(qkv, cos, sin, cu, H, 32)
    _check_stream(stream, qkv.device)
    code = {torch.float16: PK_F16, torch.bfloat16: PK_BF16}.get(op_dtype)
    if code is None:
        raise TypeError("op_dtype must be torch.float16 or torch.bfloat16")
    T = qkv.shape[0]
    with torch.cuda.device(qkv.device):
        _check_table_rows(cu, cos.shape[0], max_len)
        if out is None:
            out = torch.empty((T, H * 64), dtype=torch.float32, device=qkv.device)
        else:
            _need(out, (T, H * 64), torch.float32, "out")
        if lse is None:
            lse = torch.empty((H, T), dtype=torch.float32, device=qkv.device)
        else:
            _need(lse, (H, T), torch.float32, "lse")
        _same_device(qkv, out, lse)
        rc = pk_attend_mixed_ops(code, qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(),
                                 cu.shape[0] - 1, T, H, window, float(scale), out.data_ptr(), lse.data_ptr(),
                                 _stream_handle(stream))
        _check(rc, "pk_attend_mixed_ops")
    return out, lse


def pk_attend_tuned(dtype, qkv, cos, sin, cu, S, T, H, window, scale, longest, out, lse, stream) -> int:
    """The forward pass at the fastest usable kernel for the shape, tuned once per key (see
    include/pk.h)."""
    return load().pk_attend_tuned(dtype, qkv, cos, sin, cu, S, T, H, window, scale, longest, out, lse, stream)


def pk_tune_pick(dtype, H, window, T, longest) -> int:
    return load().pk_tune_pick(dtype, H, window, T, longest)


def pk_tune_key(dtype, H, window, T, longest) -> str:
    buf = ctypes.create_string_buffer(128)
    _check(load().pk_tune_key(dtype, H, window, T, longest, buf, 128), "pk_tune_key")
    return buf.value.decode()


def pk_tune_clear() -> int:
    return load().pk_tune_clear()


def pk_forward_kernel(dtype, window) -> int:
    return load().pk_forward_kernel(dtype, window)


def pk_kernel_name(kernel) -> str:
    return load().pk_kernel_name(kernel).decode()


def pk_attend_backward(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, dout, dqkv, stream) -> int:
    """The backward pass (see include/pk.h)."""
    return load().pk_attend_backward(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, dout, dqkv, stream)


def pk_attend_mixed(out_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream) -> int:
    """fp32 inputs and arithmetic, out in out_dtype (see include/pk.h)."""
    return load().pk_attend_mixed(out_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream)


def pk_rope(dtype, x, y, cos, sin, P, cu, S, T, H, dims, traditional, inverse, status, stream) -> int:
    """The standalone rotation of the q and k head vectors of a packed qkv (see include/pk.h)."""
    return load().pk_rope(dtype, x, y, cos, sin, P, cu, S, T, H, dims, traditional, inverse, status, stream)


def pk_schedule(cu, S, T, window, tiles, cap, stream):
    nt = ctypes.c_int64(0)
    rc = load().pk_schedule(cu, S, T, window, tiles, cap, ctypes.byref(nt), stream)
    return rc, nt.value


def pk_last_status(stream) -> int:
    return load().pk_last_status(stream)


# ------------------------------------------------------------------------------------------
# torch-tensor front (torch only allocates and supplies the stream)


def _torch():
    import torch

    return torch


def dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: PK_F32, torch.bfloat16: PK_BF16, torch.float16: PK_F16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _need(t, shape, dtype, what):
    """A caller's buffer must have exactly this shape and dtype and be a contiguous CUDA tensor:
    the C ABI receives only its address and writes the sizes the call implies."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{what} must be {tuple(shape)} {dtype}, not {tuple(t.shape)} {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")


def _check_inputs(qkv, cos, sin, cu, H, half):
    """qkv [T, 3*H*64], cos/sin [P, half] of qkv's dtype, cu [S+1] int32/uint32; all contiguous
    CUDA tensors on one device."""
    torch = _torch()
    if qkv.dim() != 2 or qkv.shape[1] != 3 * H * 64:
        raise ValueError("qkv must be [T, 3*H*64]")
    if cos.dtype != qkv.dtype or sin.dtype != qkv.dtype or cos.shape != sin.shape:
        raise TypeError("cos/sin must have qkv's dtype and one shape")
    if cos.dim() != 2 or cos.shape[1] != half:
        raise ValueError(f"cos/sin must be [P, {half}]")
    if cu.dim() != 1 or cu.dtype not in (torch.int32, torch.uint32):
        raise TypeError("cu must be a 1-D int32 or uint32 tensor")
    for t in (qkv, cos, sin, cu):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    _same_device(qkv, cos, sin, cu)


def _same_device(first, *rest):
    """Every tensor on the device of the first: the library launches on one device and
    dereferences every address there."""
    for t in rest:
        if t.device != first.device:
            raise ValueError(f"tensors on different devices ({first.device} and {t.device})")


def _check_stream(stream, device):
    """A torch stream given for the call must belong to the tensors' device."""
    dev = getattr(stream, "device", None)
    if dev is not None and dev != device:
        raise ValueError(f"stream of {dev} for tensors on {device}")


def _check_table_rows(cu, rows: int, max_len):
    """The tables must hold a row for every in-sequence position: rows >= the longest sequence.
    Without max_len this reads the longest length back from the device (one reduction and a
    synchronisation; skipped while a CUDA graph is being captured, where the caller vouches
    for the tables)."""
    torch = _torch()
    if max_len is None:
        if cu.shape[0] < 2 or (cu.is_cuda and torch.cuda.is_current_stream_capturing()):
            return
        max_len = int((cu[1:].to(torch.int64) - cu[:-1].to(torch.int64)).max().item())
    if int(max_len) > rows:
        raise ValueError(f"cos/sin hold {rows} positions but a sequence has {int(max_len)} tokens")


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def attend(qkv, cos, sin, cu, H: int, window: int, scale: float, out=None, lse=None, stream=None,
           out_dtype=None, max_len=None, tuned=False):
    """out [T, H*64] (qkv's dtype) and lse [H, T] float32 for device tensors qkv [T, 3*H*64],
    cos/sin [P, 32] (qkv's dtype) and cu [S+1] (int32 or uint32), all on one device. For
    float32 inputs, out_dtype=torch.float16 or torch.bfloat16 gives a 16-bit out
    (pk_attend_mixed). max_len: the longest sequence's length, if the caller knows it
    (otherwise it is read back from cu to check that the tables are long enough).
    tuned=True: pk_attend_tuned (the fastest usable kernel for the shape, tuned on the
    first call of each key; that call synchronizes the stream)."""
    torch = _torch()
    _check_inputs(qkv, cos, sin, cu, H, 32)
    _check_stream(stream, qkv.device)
    with torch.cuda.device(qkv.device):
        if tuned and max_len is None:
            max_len = _longest(cu)
        _check_table_rows(cu, cos.shape[0], max_len)
        return _attend(qkv, cos, sin, cu, H, window, scale, out, lse, stream, out_dtype,
                       max_len if tuned else None)


def _longest(cu) -> int:
    torch = _torch()
    if cu.shape[0] < 2:
        return 0
    return int((cu[1:].to(torch.int64) - cu[:-1].to(torch.int64)).max().item())


def _attend(qkv, cos, sin, cu, H, window, scale, out, lse, stream, out_dtype, tuned_longest=None):
    torch = _torch()
    T = qkv.shape[0]
    S = cu.shape[0] - 1
    # the output type: out_dtype, else a given out's, else qkv's
    odt = out_dtype if out_dtype is not None else (out.dtype if out is not None else qkv.dtype)
    if odt != qkv.dtype and qkv.dtype != torch.float32:
        raise TypeError("a different output type needs float32 inputs")
    if out is None:
        out = torch.empty((T, H * 64), dtype=odt, device=qkv.device)
    else:
        _need(out, (T, H * 64), odt, "out")
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=qkv.device)
    else:
        _need(lse, (H, T), torch.float32, "lse")
    _same_device(qkv, out, lse)
    if tuned_longest is not None and odt != qkv.dtype:
        raise TypeError("the tuned entry point writes out in qkv's type")
    if tuned_longest is not None:
        rc = pk_attend_tuned(dtype_code(qkv), qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(),
                             S, T, H, window, float(scale), int(tuned_longest), out.data_ptr(), lse.data_ptr(),
                             _stream_handle(stream))
    elif odt != qkv.dtype:
        rc = pk_attend_mixed(dtype_code(out), qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(),
                             S, T, H, window, float(scale), out.data_ptr(), lse.data_ptr(), _stream_handle(stream))
    else:
        rc = pk_attend_dt(dtype_code(qkv), qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(),
                          S, T, H, window, float(scale), out.data_ptr(), lse.data_ptr(),
                          _stream_handle(stream))
    _check(rc, "pk_attend")
    return out, lse


def attend_backward(qkv, cos, sin, cu, H: int, window: int, scale: float, out, lse, dout, dqkv=None, stream=None,
                    max_len=None):
    """dqkv [T, 3*H*64] (qkv's dtype): the gradient of sum(dout * out) with respect to qkv, for
    the forward's out and lse (max_len as for attend)."""
    torch = _torch()
    T = qkv.shape[0]
    S = cu.shape[0] - 1
    _check_inputs(qkv, cos, sin, cu, H, 32)
    _need(out, (T, H * 64), qkv.dtype, "out")
    _need(dout, (T, H * 64), qkv.dtype, "dout")
    _need(lse, (H, T), torch.float32, "lse")
    if dqkv is not None:
        _need(dqkv, tuple(qkv.shape), qkv.dtype, "dqkv")
        _same_device(qkv, dqkv)
    _same_device(qkv, out, lse, dout)
    _check_stream(stream, qkv.device)
    with torch.cuda.device(qkv.device):
        _check_table_rows(cu, cos.shape[0], max_len)
        if dqkv is None:
            dqkv = torch.empty_like(qkv)
        return _attend_backward(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, dout, dqkv, stream)


def _attend_backward(qkv, cos, sin, cu, S, T, H, window, scale, out, lse, dout, dqkv, stream):
    rc = pk_attend_backward(dtype_code(qkv), qkv.data_ptr(), cos.data_ptr(), sin.data_ptr(), cu.data_ptr(), S, T, H,
                            window, float(scale), out.data_ptr(), lse.data_ptr(), dout.data_ptr(), dqkv.data_ptr(),
                            _stream_handle(stream))
    _check(rc, "pk_attend_backward")
    return dqkv


def rope(qkv, cos, sin, cu, H: int, dims: int = 64, traditional: bool = False, inverse: bool = False,
         out=None, status=None, stream=None):
    """qkv [T, 3*H*64] with the first `dims` features of every q and k head vector rotated at
    their in-sequence positions (tables cos/sin [P, dims/2] in qkv's dtype); v copied. `out`
    may be qkv itself (in place). `status`: optional int32 device tensor of one element."""
    torch = _torch()
    T = qkv.shape[0]
    S = cu.shape[0] - 1
    _check_inputs(qkv, cos, sin, cu, H, dims // 2)
    _check_stream(stream, qkv.device)
    if out is None:
        out = torch.empty_like(qkv)
    else:
        _need(out, tuple(qkv.shape), qkv.dtype, "out")
        _same_device(qkv, out)
    if status is not None:
        _need(status, (1,), torch.int32, "status")
        _same_device(qkv, status)
    with torch.cuda.device(qkv.device):
        return _rope(qkv, cos, sin, cu, S, T, H, dims, traditional, inverse, out, status, stream)


def _rope(qkv, cos, sin, cu, S, T, H, dims, traditional, inverse, out, status, stream):
    rc = pk_rope(dtype_code(qkv), qkv.data_ptr(), out.data_ptr(), cos.data_ptr(), sin.data_ptr(),
                 cos.shape[0], cu.data_ptr(), S, T, H, int(dims), int(bool(traditional)), int(bool(inverse)),
                 status.data_ptr() if status is not None else None, _stream_handle(stream))
    _check(rc, "pk_rope")
    return out


def schedule(cu, T: int, window: int, stream=None):
    """Tile records [NT, 8] (int32 tensor holding the uint32 fields) of the device scheduler."""
    torch = _torch()
    if cu.dim() != 1 or cu.dtype not in (torch.int32, torch.uint32) or not cu.is_cuda or not cu.is_contiguous():
        raise ValueError("cu must be a contiguous 1-D int32 or uint32 CUDA tensor")
    cap = int(load().pk_schedule_capacity(T))
    tiles = torch.zeros((max(cap, 1), 8), dtype=torch.int32, device=cu.device)
    rc, nt = pk_schedule(cu.data_ptr(), cu.shape[0] - 1, T, window, tiles.data_ptr(), cap,
                         _stream_handle(stream))
    _check(rc, "pk_schedule")
    return tiles[:nt]


def last_status(stream=None) -> int:
    return pk_last_status(_stream_handle(stream))


def profile_start(n: int):
    """Record kernel events around the next n attention calls (see pk_profile_start)."""
    _check(load().pk_profile_start(int(n)), "pk_profile_start")


def profile_stop():
    """(schedule_ms_total, attend_ms_total, calls) recorded since profile_start."""
    a, b, n = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int(0)
    _check(load().pk_profile_stop(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n)), "pk_profile_stop")
    return a.value, b.value, n.value


def release():
    _check(load().pk_release(), "pk_release")
