"""Python binding of libmfx, fused transformer MLP and residual epilogues for
GB300 (sm_103a).

Every function here marshals torch tensors into the C ABI declared in
``include/mfx.h`` (device pointers, sizes, the current CUDA stream) and calls
the library; all computation happens in its CUDA kernels.  The names are the
ABI's names and the positional arguments follow the ABI's order.  Tensors must
be contiguous CUDA tensors; the last dimension is the width (hidden, or 2F for
the GLU inputs) and all leading dimensions are flattened into rows, so the
Megatron [seq, batch, hidden] layout is accepted as is.

There is no fallback: if ``libmfx.so`` has not been built, every call raises.
"""
import ctypes as C
import os

import torch

__all__ = [
    "MfxError", "lib", "dtype_code",
    "mfx_bias_gelu_fwd", "mfx_bias_gelu_bwd",
    "mfx_bias_geglu_fwd", "mfx_bias_geglu_bwd",
    "mfx_bias_swiglu_fwd", "mfx_bias_swiglu_bwd",
    "mfx_weighted_squared_relu_fwd", "mfx_weighted_squared_relu_bwd",
    "mfx_scaled_masked_softmax_fwd", "mfx_scaled_upper_triang_masked_softmax_fwd",
    "mfx_scaled_masked_softmax_bwd", "mfx_scaled_upper_triang_masked_softmax_bwd",
    "mfx_bias_dropout_add_train", "mfx_bias_dropout_add_inference", "mfx_bias_dropout_add_bwd",
    "mfx_bias_dropout_add_train_packed", "mfx_bias_dropout_add_bwd_packed",
    "mfx_bias_gelu_bwd_dbias", "mfx_bias_geglu_bwd_dbias", "mfx_bias_swiglu_bwd_dbias",
    "mfx_bias_dropout_add_bwd_dbias", "mfx_device_error",
]

# MFX_LIBRARY selects another build of the same library (for example one
# compiled with different tuning knobs); by default the in-tree build is used.
LIB_PATH = os.environ.get("MFX_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libmfx.so")

MFX_F32, MFX_BF16 = 0, 1
STATUS = {0: "MFX_OK", 1: "MFX_ERR_NULL", 2: "MFX_ERR_SHAPE", 3: "MFX_ERR_DTYPE",
          4: "MFX_ERR_PROB", 5: "MFX_ERR_ALIAS", 6: "MFX_ERR_CUDA", 7: "MFX_ERR_DEVICE",
          8: "MFX_ERR_WORKSPACE"}


class MfxError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().mfx_status_string(status).decode()
        extra = f" (cudaError {lib().mfx_last_cuda_error()})" if status == 6 else ""
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}{extra}")


_lib = None

_P, _I, _I64, _U64, _F = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float
_SIGS = {
    "mfx_bias_gelu_fwd": [_I, _I64, _I64, _P, _P, _P, _P],
    "mfx_bias_gelu_bwd": [_I, _I64, _I64, _P, _P, _P, _P, _P],
    "mfx_bias_geglu_fwd": [_I, _I64, _I64, _P, _P, _P, _P],
    "mfx_bias_geglu_bwd": [_I, _I64, _I64, _P, _P, _P, _P, _P],
    "mfx_bias_swiglu_fwd": [_I, _I64, _I64, _P, _P, _P, _P, _P],
    "mfx_bias_swiglu_bwd": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P, _P],
    "mfx_weighted_squared_relu_fwd": [_I, _I64, _I64, _P, _P, _P, _P],
    "mfx_weighted_squared_relu_bwd": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P],
    "mfx_scaled_masked_softmax_fwd": [_I, _I64, _I64, _I64, _I64, _P, _P, _I64, _I64, _I64, _F, _P, _P],
    "mfx_scaled_upper_triang_masked_softmax_fwd": [_I, _I64, _I64, _P, _F, _P, _P],
    "mfx_scaled_masked_softmax_bwd": [_I, _I64, _I64, _P, _P, _F, _P, _P],
    "mfx_scaled_upper_triang_masked_softmax_bwd": [_I, _I64, _I64, _P, _P, _F, _P, _P],
    "mfx_bias_dropout_add_train": [_I, _I, _I64, _I64, _P, _P, _P, _F, _U64, _U64, _U64, _P, _P, _P],
    "mfx_bias_dropout_add_inference": [_I, _I, _I64, _I64, _P, _P, _P, _F, _U64, _U64, _P],
    "mfx_bias_dropout_add_bwd": [_I, _I, _I64, _I64, _P, _P, _F, _U64, _U64, _U64, _P, _P, _P],
    "mfx_bias_dropout_add_train_packed": [_I, _I, _I64, _I64, _P, _P, _P, _F, _U64, _U64, _U64, _P, _P, _P],
    "mfx_bias_dropout_add_bwd_packed": [_I, _I, _I64, _I64, _P, _P, _F, _P, _P, _P],
    "mfx_bias_gelu_bwd_dbias": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P, C.POINTER(C.c_size_t), _P],
    "mfx_bias_gelu_bwd_dbias_noalloc": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P],
    "mfx_bias_geglu_bwd_dbias": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P, C.POINTER(C.c_size_t), _P],
    "mfx_bias_swiglu_bwd_dbias": [_I, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, C.POINTER(C.c_size_t), _P],
    "mfx_bias_dropout_add_bwd_dbias": [_I, _I, _I64, _I64, _P, _P, _F, _U64, _U64, _U64, _P, _P, _P, _P,
                                       C.POINTER(C.c_size_t), _P],
}


def lib():
    """The loaded libmfx.so (ctypes), with argument types set."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libmfx.so is not built ({LIB_PATH} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = C.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        L.mfx_status_string.argtypes = [C.c_int]
        L.mfx_status_string.restype = C.c_char_p
        L.mfx_last_cuda_error.argtypes = []
        L.mfx_last_cuda_error.restype = C.c_int
        L.mfx_version.argtypes = []
        L.mfx_version.restype = C.c_int
        L.mfx_device_error.argtypes = [C.POINTER(C.c_uint)]
        L.mfx_device_error.restype = C.c_int
        _lib = L
    return _lib


def dtype_code(dtype):
    if dtype == torch.bfloat16:
        return MFX_BF16
    if dtype == torch.float32:
        return MFX_F32
    raise TypeError(f"libmfx supports bfloat16 and float32 tensors, got {dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _cuda(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


# the current stream's raw handle without building a Stream object per call
# (torch's own raw-stream query where this torch has it)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, t):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(t.get_device())
        return torch.cuda.current_stream(t.device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _rows_cols(t):
    cols = t.shape[-1] if t.dim() else 1
    rows = t.numel() // cols if cols else 0
    return rows, cols


def mfx_device_error():
    """Code of any bounded wait that ran out since the last call (0 = none);
    synchronises the current device and clears the word."""
    code = C.c_uint(0)
    lib().mfx_device_error(C.byref(code))
    return code.value


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise MfxError(st, name)


# ---------------------------------------------------------------------------
# bias-GeLU
# ---------------------------------------------------------------------------
def mfx_bias_gelu_fwd(bias, y, out=None, stream=None):
    """out = gelu_tanh(y + bias); returns out (allocated if not given)."""
    _cuda(y, "y")
    _cuda(bias, "bias", y.dtype)
    out = torch.empty_like(y) if out is None else _cuda(out, "out", y.dtype)
    rows, cols = _rows_cols(y)
    _call("mfx_bias_gelu_fwd", dtype_code(y.dtype), rows, cols, _ptr(bias), _ptr(y), _ptr(out),
          _stream(stream, y))
    return out


def mfx_bias_gelu_bwd(g, bias, y, dy=None, stream=None):
    """dy = g * gelu_tanh'(y + bias); returns dy."""
    _cuda(y, "y")
    _cuda(g, "g", y.dtype)
    _cuda(bias, "bias", y.dtype)
    if g.shape != y.shape:
        raise ValueError("g and y must have the same shape")
    dy = torch.empty_like(y) if dy is None else _cuda(dy, "dy", y.dtype)
    rows, cols = _rows_cols(y)
    _call("mfx_bias_gelu_bwd", dtype_code(y.dtype), rows, cols, _ptr(g), _ptr(bias), _ptr(y),
          _ptr(dy), _stream(stream, y))
    return dy


# ---------------------------------------------------------------------------
# GLU
# ---------------------------------------------------------------------------
def _glu_shape(x):
    rows, two_f = _rows_cols(x)
    if two_f % 2:
        raise ValueError("the GLU input width must be even (2F)")
    return rows, two_f // 2


def _half_shape(x):
    return (*x.shape[:-1], x.shape[-1] // 2)


def mfx_bias_geglu_fwd(x, bias, out=None, stream=None):
    _cuda(x, "x")
    _cuda(bias, "bias", x.dtype)
    rows, F = _glu_shape(x)
    out = x.new_empty(_half_shape(x)) if out is None else _cuda(out, "out", x.dtype)
    _call("mfx_bias_geglu_fwd", dtype_code(x.dtype), rows, F, _ptr(x), _ptr(bias), _ptr(out),
          _stream(stream, x))
    return out


def mfx_bias_geglu_bwd(g, x, bias, dx=None, stream=None):
    _cuda(x, "x")
    _cuda(g, "g", x.dtype)
    _cuda(bias, "bias", x.dtype)
    rows, F = _glu_shape(x)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx", x.dtype)
    _call("mfx_bias_geglu_bwd", dtype_code(x.dtype), rows, F, _ptr(g), _ptr(x), _ptr(bias),
          _ptr(dx), _stream(stream, x))
    return dx


def mfx_bias_swiglu_fwd(x, bias, weight=None, out=None, stream=None):
    _cuda(x, "x")
    _cuda(bias, "bias", x.dtype)
    _cuda(weight, "weight", torch.float32)
    rows, F = _glu_shape(x)
    out = x.new_empty(_half_shape(x)) if out is None else _cuda(out, "out", x.dtype)
    _call("mfx_bias_swiglu_fwd", dtype_code(x.dtype), rows, F, _ptr(x), _ptr(bias), _ptr(weight),
          _ptr(out), _stream(stream, x))
    return out


def mfx_bias_swiglu_bwd(g, x, bias, weight=None, dx=None, dweight=None, stream=None):
    """Returns (dx, dweight); dweight is None without a weight."""
    _cuda(x, "x")
    _cuda(g, "g", x.dtype)
    _cuda(bias, "bias", x.dtype)
    _cuda(weight, "weight", torch.float32)
    rows, F = _glu_shape(x)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx", x.dtype)
    if weight is not None and dweight is None:
        dweight = torch.empty(weight.shape, dtype=torch.float32, device=x.device)
    _cuda(dweight, "dweight", torch.float32)
    _call("mfx_bias_swiglu_bwd", dtype_code(x.dtype), rows, F, _ptr(g), _ptr(x), _ptr(bias),
          _ptr(weight), _ptr(dx), _ptr(dweight), _stream(stream, x))
    return dx, dweight


# ---------------------------------------------------------------------------
# weighted squared ReLU
# ---------------------------------------------------------------------------
def _row_weight(weight, rows):
    _cuda(weight, "weight", torch.float32)
    if weight is None or weight.numel() != rows:
        raise ValueError(f"weight must be a float32 CUDA tensor of {rows} elements (one per row)")
    return weight


def mfx_weighted_squared_relu_fwd(x, weight, out=None, stream=None):
    _cuda(x, "x")
    rows, cols = _rows_cols(x)
    _row_weight(weight, rows)
    out = torch.empty_like(x) if out is None else _cuda(out, "out", x.dtype)
    _call("mfx_weighted_squared_relu_fwd", dtype_code(x.dtype), rows, cols, _ptr(x), _ptr(weight),
          _ptr(out), _stream(stream, x))
    return out


def mfx_weighted_squared_relu_bwd(g, x, weight, dx=None, dweight=None, stream=None):
    """Returns (dx, dweight)."""
    _cuda(x, "x")
    _cuda(g, "g", x.dtype)
    rows, cols = _rows_cols(x)
    _row_weight(weight, rows)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx", x.dtype)
    if dweight is None:
        dweight = torch.empty(weight.shape, dtype=torch.float32, device=x.device)
    _cuda(dweight, "dweight", torch.float32)
    _call("mfx_weighted_squared_relu_bwd", dtype_code(x.dtype), rows, cols, _ptr(g), _ptr(x), _ptr(weight),
          _ptr(dx), _ptr(dweight), _stream(stream, x))
    return dx, dweight


# ---------------------------------------------------------------------------
# scale-mask-softmax
# ---------------------------------------------------------------------------
def mfx_scaled_masked_softmax_fwd(x, scale, mask=None, y=None, stream=None):
    """Softmax over the last dim of x * scale (+ mask).  x: [b, np, sq, sk]
    (or any shape whose leading dims flatten into rows when mask is None);
    mask: additive, 4 dims [1|b, 1|np, 1|sq, sk], x's dtype."""
    _cuda(x, "x")
    _cuda(mask, "mask", x.dtype)
    if mask is not None:
        if x.dim() != 4 or mask.dim() != 4:
            raise ValueError("with a mask, x and mask must have 4 dims [b, np, sq, sk]")
        b, np_, sq, sk = x.shape
        mb, mnp, msq, msk = mask.shape
    else:
        sk = x.shape[-1] if x.dim() else 1
        b, np_, sq = 1, 1, (x.numel() // sk if sk else 0)
        mb = mnp = msq = 1
        msk = sk
    if msk != sk:
        raise ValueError("mask's last dim must equal x's")
    y = torch.empty_like(x) if y is None else _cuda(y, "y", x.dtype)
    _call("mfx_scaled_masked_softmax_fwd", dtype_code(x.dtype), b, np_, sq, sk, _ptr(x), _ptr(mask),
          mb, mnp, msq, float(scale), _ptr(y), _stream(stream, x))
    return y


def _causal_dims(t):
    if t.dim() != 3 or t.shape[1] != t.shape[2]:
        raise ValueError("the causal softmax takes [attn_batches, sq, sq]")
    return t.shape[0], t.shape[1]


def mfx_scaled_upper_triang_masked_softmax_fwd(x, scale, y=None, stream=None):
    _cuda(x, "x")
    ab, sq = _causal_dims(x)
    y = torch.empty_like(x) if y is None else _cuda(y, "y", x.dtype)
    _call("mfx_scaled_upper_triang_masked_softmax_fwd", dtype_code(x.dtype), ab, sq, _ptr(x), float(scale),
          _ptr(y), _stream(stream, x))
    return y


def mfx_scaled_masked_softmax_bwd(dy, y, scale, dx=None, stream=None):
    _cuda(y, "y")
    _cuda(dy, "dy", y.dtype)
    if dy.shape != y.shape:
        raise ValueError("dy and y must have the same shape")
    rows, sk = _rows_cols(y)
    dx = torch.empty_like(y) if dx is None else _cuda(dx, "dx", y.dtype)
    _call("mfx_scaled_masked_softmax_bwd", dtype_code(y.dtype), rows, sk, _ptr(dy), _ptr(y), float(scale),
          _ptr(dx), _stream(stream, y))
    return dx


def mfx_scaled_upper_triang_masked_softmax_bwd(dy, y, scale, dx=None, stream=None):
    _cuda(y, "y")
    _cuda(dy, "dy", y.dtype)
    if dy.shape != y.shape:
        raise ValueError("dy and y must have the same shape")
    ab, sq = _causal_dims(y)
    dx = torch.empty_like(y) if dx is None else _cuda(dx, "dx", y.dtype)
    _call("mfx_scaled_upper_triang_masked_softmax_bwd", dtype_code(y.dtype), ab, sq, _ptr(dy), _ptr(y),
          float(scale), _ptr(dx), _stream(stream, y))
    return dx


# ---------------------------------------------------------------------------
# bias-dropout-add
# ---------------------------------------------------------------------------
def mfx_bias_dropout_add_train(x, bias, residual, p, seed, offset=0, elem_base=0, out=None,
                               keep_mask=None, stream=None):
    """Returns (out, keep_mask); keep_mask is uint8 (1 = kept)."""
    _cuda(x, "x")
    _cuda(bias, "bias", x.dtype)
    _cuda(residual, "residual")
    if residual.shape != x.shape:
        raise ValueError("residual must have x's shape")
    out = torch.empty_like(x) if out is None else _cuda(out, "out", x.dtype)
    keep_mask = (torch.empty(x.shape, dtype=torch.uint8, device=x.device) if keep_mask is None
                 else _cuda(keep_mask, "keep_mask", torch.uint8))
    rows, cols = _rows_cols(x)
    _call("mfx_bias_dropout_add_train", dtype_code(x.dtype), dtype_code(residual.dtype), rows, cols,
          _ptr(x), _ptr(bias), _ptr(residual), float(p), int(seed) % 2**64, int(offset) % 2**64,
          int(elem_base), _ptr(out), _ptr(keep_mask), _stream(stream, x))
    return out, keep_mask


def mfx_bias_dropout_add_inference(x, bias, residual, p=0.0, seed=0, offset=0, stream=None):
    """x = (x + bias) + residual.to(x.dtype), in place; returns x."""
    _cuda(x, "x")
    _cuda(bias, "bias", x.dtype)
    _cuda(residual, "residual")
    if residual.shape != x.shape:
        raise ValueError("residual must have x's shape")
    rows, cols = _rows_cols(x)
    _call("mfx_bias_dropout_add_inference", dtype_code(x.dtype), dtype_code(residual.dtype), rows,
          cols, _ptr(x), _ptr(bias), _ptr(residual), float(p), int(seed) % 2**64,
          int(offset) % 2**64, _stream(stream, x))
    return x


def mfx_bias_dropout_add_bwd(g, keep_mask, p, seed=0, offset=0, elem_base=0, dx=None, dresidual=None,
                             residual_dtype=None, stream=None):
    """Returns (dx, dresidual).  keep_mask None regenerates the forward's mask
    from (seed, offset, elem_base, p).  dresidual is produced when a buffer
    is given or residual_dtype is set (and differs from g's dtype; with the
    same dtype the residual gradient is g itself)."""
    _cuda(g, "g")
    _cuda(keep_mask, "keep_mask", torch.uint8)
    dx = torch.empty_like(g) if dx is None else _cuda(dx, "dx", g.dtype)
    if dresidual is None and residual_dtype is not None:
        dresidual = g if residual_dtype == g.dtype else torch.empty(g.shape, dtype=residual_dtype,
                                                                     device=g.device)
    _cuda(dresidual, "dresidual")
    rdt = dtype_code(dresidual.dtype) if dresidual is not None else dtype_code(g.dtype)
    rows, cols = _rows_cols(g)
    _call("mfx_bias_dropout_add_bwd", dtype_code(g.dtype), rdt, rows, cols, _ptr(g), _ptr(keep_mask),
          float(p), int(seed) % 2**64, int(offset) % 2**64, int(elem_base), _ptr(dx), _ptr(dresidual),
          _stream(stream, g))
    return dx, dresidual


def mfx_bias_dropout_add_train_packed(x, bias, residual, p, seed, offset=0, elem_base=0, out=None,
                                      keep_bits=None, stream=None):
    """Returns (out, keep_bits): the keep mask as bits, element i at bit i % 8
    of byte i // 8 (uint8, ceil(numel / 8) bytes)."""
    _cuda(x, "x")
    _cuda(bias, "bias", x.dtype)
    _cuda(residual, "residual")
    if residual.shape != x.shape:
        raise ValueError("residual must have x's shape")
    out = torch.empty_like(x) if out is None else _cuda(out, "out", x.dtype)
    nbytes = (x.numel() + 7) // 8
    keep_bits = (torch.empty(nbytes, dtype=torch.uint8, device=x.device) if keep_bits is None
                 else _cuda(keep_bits, "keep_bits", torch.uint8))
    if keep_bits.numel() < nbytes:
        raise ValueError(f"keep_bits needs {nbytes} bytes")
    rows, cols = _rows_cols(x)
    _call("mfx_bias_dropout_add_train_packed", dtype_code(x.dtype), dtype_code(residual.dtype), rows, cols,
          _ptr(x), _ptr(bias), _ptr(residual), float(p), int(seed) % 2**64, int(offset) % 2**64,
          int(elem_base), _ptr(out), _ptr(keep_bits), _stream(stream, x))
    return out, keep_bits


def mfx_bias_dropout_add_bwd_packed(g, keep_bits, p, dx=None, dresidual=None, residual_dtype=None, stream=None):
    """(dx, dresidual) from the bit mask of mfx_bias_dropout_add_train_packed."""
    _cuda(g, "g")
    _cuda(keep_bits, "keep_bits", torch.uint8)
    if keep_bits.numel() < (g.numel() + 7) // 8:
        raise ValueError("keep_bits is shorter than the mask")
    dx = torch.empty_like(g) if dx is None else _cuda(dx, "dx", g.dtype)
    if dresidual is None and residual_dtype is not None:
        dresidual = g if residual_dtype == g.dtype else torch.empty(g.shape, dtype=residual_dtype,
                                                                     device=g.device)
    _cuda(dresidual, "dresidual")
    rdt = dtype_code(dresidual.dtype) if dresidual is not None else dtype_code(g.dtype)
    rows, cols = _rows_cols(g)
    _call("mfx_bias_dropout_add_bwd_packed", dtype_code(g.dtype), rdt, rows, cols, _ptr(g), _ptr(keep_bits),
          float(p), _ptr(dx), _ptr(dresidual), _stream(stream, g))
    return dx, dresidual


# ---------------------------------------------------------------------------
# fused bias gradients (workspace protocol: query the size, then run)
# ---------------------------------------------------------------------------
def _with_workspace(name, args_before_ws, tail, device, workspace=None):
    """Query the workspace size, allocate it and run `name`.  `workspace` is
    None (a fresh uint8 tensor), a uint8 CUDA tensor, or a callable that
    takes the byte count and returns one (a caller's own allocator)."""
    size = C.c_size_t(0)
    _call(name, *args_before_ws, None, C.byref(size), *tail)
    if workspace is None:
        workspace = torch.empty(max(int(size.value), 16), dtype=torch.uint8, device=device)
    else:
        if callable(workspace):
            workspace = workspace(max(int(size.value), 16))
        _cuda(workspace, "workspace", torch.uint8)
    size = C.c_size_t(workspace.numel())
    _call(name, *args_before_ws, _ptr(workspace), C.byref(size), *tail)
    return workspace


def mfx_bias_gelu_bwd_dbias(g, bias, y, dy=None, dbias=None, workspace=None, stream=None):
    """(dy, dbias): bias-GeLU backward and the bias gradient sum_r dy[r, :]."""
    _cuda(y, "y")
    _cuda(g, "g", y.dtype)
    _cuda(bias, "bias", y.dtype)
    rows, cols = _rows_cols(y)
    dy = torch.empty_like(y) if dy is None else _cuda(dy, "dy", y.dtype)
    dbias = y.new_empty((cols,)) if dbias is None else _cuda(dbias, "dbias", y.dtype)
    st = _stream(stream, y)
    _with_workspace("mfx_bias_gelu_bwd_dbias",
                    (dtype_code(y.dtype), rows, cols, _ptr(g), _ptr(bias), _ptr(y), _ptr(dy), _ptr(dbias)),
                    (st,), y.device, workspace)
    return dy, dbias


def mfx_bias_gelu_bwd_dbias_noalloc(g, bias, y, dy=None, dbias=None, stream=None):
    """(dy, dbias) as mfx_bias_gelu_bwd_dbias, with the library's fixed
    device scratch instead of a caller workspace (widths up to the scratch
    size; concurrent calls on the GPU must be serialised)."""
    _cuda(y, "y")
    _cuda(g, "g", y.dtype)
    _cuda(bias, "bias", y.dtype)
    rows, cols = _rows_cols(y)
    dy = torch.empty_like(y) if dy is None else _cuda(dy, "dy", y.dtype)
    dbias = y.new_empty((cols,)) if dbias is None else _cuda(dbias, "dbias", y.dtype)
    _call("mfx_bias_gelu_bwd_dbias_noalloc", dtype_code(y.dtype), rows, cols, _ptr(g), _ptr(bias), _ptr(y),
          _ptr(dy), _ptr(dbias), _stream(stream, y))
    return dy, dbias


def mfx_bias_geglu_bwd_dbias(g, x, bias, dx=None, dbias=None, workspace=None, stream=None):
    """(dx, dbias): GEGLU backward and the bias gradient over the width 2F."""
    _cuda(x, "x")
    _cuda(g, "g", x.dtype)
    _cuda(bias, "bias", x.dtype)
    rows, F = _glu_shape(x)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx", x.dtype)
    dbias = x.new_empty((2 * F,)) if dbias is None else _cuda(dbias, "dbias", x.dtype)
    _with_workspace("mfx_bias_geglu_bwd_dbias",
                    (dtype_code(x.dtype), rows, F, _ptr(g), _ptr(x), _ptr(bias), _ptr(dx), _ptr(dbias)),
                    (_stream(stream, x),), x.device, workspace)
    return dx, dbias


def mfx_bias_swiglu_bwd_dbias(g, x, bias, weight=None, dx=None, dweight=None, dbias=None, workspace=None,
                              stream=None):
    """(dx, dweight, dbias): SwiGLU backward (optionally weighted) and the bias
    gradient over the width 2F."""
    _cuda(x, "x")
    _cuda(g, "g", x.dtype)
    _cuda(bias, "bias", x.dtype)
    _cuda(weight, "weight", torch.float32)
    rows, F = _glu_shape(x)
    dx = torch.empty_like(x) if dx is None else _cuda(dx, "dx", x.dtype)
    if weight is not None and dweight is None:
        dweight = torch.empty(weight.shape, dtype=torch.float32, device=x.device)
    dbias = x.new_empty((2 * F,)) if dbias is None else _cuda(dbias, "dbias", x.dtype)
    _with_workspace("mfx_bias_swiglu_bwd_dbias",
                    (dtype_code(x.dtype), rows, F, _ptr(g), _ptr(x), _ptr(bias), _ptr(weight), _ptr(dx),
                     _ptr(dweight), _ptr(dbias)), (_stream(stream, x),), x.device, workspace)
    return dx, dweight, dbias


def mfx_bias_dropout_add_bwd_dbias(g, keep_mask, p, seed=0, offset=0, elem_base=0, dx=None, dresidual=None,
                                   residual_dtype=None, dbias=None, workspace=None, stream=None):
    """(dx, dresidual, dbias): bias-dropout-add backward and the bias
    gradient sum_r dx[r, :]."""
    _cuda(g, "g")
    _cuda(keep_mask, "keep_mask", torch.uint8)
    dx = torch.empty_like(g) if dx is None else _cuda(dx, "dx", g.dtype)
    if dresidual is None and residual_dtype is not None:
        dresidual = g if residual_dtype == g.dtype else torch.empty(g.shape, dtype=residual_dtype,
                                                                     device=g.device)
    _cuda(dresidual, "dresidual")
    rdt = dtype_code(dresidual.dtype) if dresidual is not None else dtype_code(g.dtype)
    rows, cols = _rows_cols(g)
    dbias = g.new_empty((cols,)) if dbias is None else _cuda(dbias, "dbias", g.dtype)
    _with_workspace("mfx_bias_dropout_add_bwd_dbias",
                    (dtype_code(g.dtype), rdt, rows, cols, _ptr(g), _ptr(keep_mask), float(p),
                     int(seed) % 2**64, int(offset) % 2**64, int(elem_base), _ptr(dx), _ptr(dresidual),
                     _ptr(dbias)), (_stream(stream, g),), g.device, workspace)
    return dx, dresidual, dbias
