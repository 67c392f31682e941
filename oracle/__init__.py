"""ctypes front end of the CPU oracle (``oracle/mfx_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package; the library and
its Python binding never do.  Arrays are numpy: bf16 tensors travel as their
raw ``uint16`` bit patterns, fp32 as ``float32``; activation results come back
as ``float64``.
"""
import ctypes as C

import numpy as np

from .build import build

F32, BF16 = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        P, I64, U64, F, D = C.c_void_p, C.c_int64, C.c_uint64, C.c_float, C.c_double
        sig = {
            "orc_bf16_to_f32": (F, [C.c_uint16]),
            "orc_f32_to_bf16": (C.c_uint16, [F]),
            "orc_gelu_tanh": (D, [D]),
            "orc_gelu_tanh_grad": (D, [D]),
            "orc_logistic": (D, [D]),
            "orc_silu": (D, [D]),
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_philox4x64_10": (None, [P, P, P]),
            "orc_philox4x32_rounds": (None, [C.c_int, P, P, P]),
            "orc_dropout_threshold": (C.c_uint32, [F]),
            "orc_uniform16": (C.c_uint32, [U64, U64, U64]),
            "orc_keep_mask": (None, [U64, U64, U64, I64, F, P]),
            "orc_bias_gelu_fwd": (None, [C.c_int, I64, I64, P, P, P]),
            "orc_bias_gelu_bwd": (None, [C.c_int, I64, I64, P, P, P, P, P]),
            "orc_bias_geglu_fwd": (None, [C.c_int, I64, I64, P, P, P]),
            "orc_bias_geglu_bwd": (None, [C.c_int, I64, I64, P, P, P, P, P]),
            "orc_bias_swiglu_fwd": (None, [C.c_int, I64, I64, P, P, P, P]),
            "orc_bias_swiglu_bwd": (None, [C.c_int, I64, I64, P, P, P, P, P, P, P, P]),
            "orc_bias_dropout_add_train": (None, [C.c_int, C.c_int, I64, I64, P, P, P, F,
                                                  U64, U64, U64, P, P]),
            "orc_bias_dropout_add_inference": (None, [C.c_int, C.c_int, I64, I64, P, P, P]),
            "orc_bias_dropout_add_bwd": (None, [C.c_int, C.c_int, I64, I64, P, P, F, U64, U64, U64, P, P]),
            "orc_column_sums": (None, [C.c_int, I64, I64, P, P, P]),
            "orc_weighted_squared_relu_fwd": (None, [C.c_int, I64, I64, P, P, P]),
            "orc_weighted_squared_relu_bwd": (None, [C.c_int, I64, I64, P, P, P, P, P, P]),
            "orc_scaled_masked_softmax_fwd": (None, [C.c_int, I64, I64, I64, I64, P, P, I64, I64, I64,
                                                     C.c_int, F, P]),
            "orc_scaled_softmax_bwd": (None, [C.c_int, I64, I64, P, P, C.c_int, F, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _dt(a):
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes uint16 (bf16 bits) or float32, got {a.dtype}")


# ---- scalar pieces ---------------------------------------------------------
def gelu_tanh(x):
    return np.array([lib().orc_gelu_tanh(float(v)) for v in np.ravel(x)]).reshape(np.shape(x))


def gelu_tanh_grad(x):
    return np.array([lib().orc_gelu_tanh_grad(float(v)) for v in np.ravel(x)]).reshape(np.shape(x))


def logistic(z):
    return np.array([lib().orc_logistic(float(v)) for v in np.ravel(z)]).reshape(np.shape(z))


def silu(z):
    return np.array([lib().orc_silu(float(v)) for v in np.ravel(z)]).reshape(np.shape(z))


def bf16_bits_from_f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    f = lib().orc_f32_to_bf16
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def f32_from_bf16_bits(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    f = lib().orc_bf16_to_f32
    return np.array([f(int(v)) for v in h.ravel()], dtype=np.float32).reshape(h.shape)


def philox4x32_10(ctr, key, rounds=10):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_rounds(rounds, _ptr(c), _ptr(k), _ptr(out))
    return out


def philox4x64_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    lib().orc_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def dropout_threshold(p):
    return int(lib().orc_dropout_threshold(float(p)))


def uniform16(seed, offset, e):
    return int(lib().orc_uniform16(seed, offset, e))


def keep_mask(seed, offset, elem_base, n, p):
    out = np.zeros(n, dtype=np.uint8)
    lib().orc_keep_mask(seed, offset, elem_base, n, float(p), _ptr(out))
    return out


# ---- tensor ops --------------------------------------------------------------
def bias_gelu_fwd(y, bias=None):
    y = np.ascontiguousarray(y)
    rows, cols = y.shape
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_bias_gelu_fwd(_dt(y), rows, cols, _ptr(bias), _ptr(y), _ptr(out))
    return out


def bias_gelu_bwd(g, y, bias=None, with_scale=False):
    """dy, or (dy, scale) with the per-element condition scale."""
    y = np.ascontiguousarray(y)
    g = np.ascontiguousarray(g)
    assert g.dtype == y.dtype and g.shape == y.shape
    rows, cols = y.shape
    out = np.empty((rows, cols), dtype=np.float64)
    scale = np.empty((rows, cols), dtype=np.float64) if with_scale else None
    lib().orc_bias_gelu_bwd(_dt(y), rows, cols, _ptr(g), _ptr(bias), _ptr(y), _ptr(out), _ptr(scale))
    return (out, scale) if with_scale else out


def bias_geglu_fwd(x, bias=None):
    x = np.ascontiguousarray(x)
    rows, two_f = x.shape
    F = two_f // 2
    out = np.empty((rows, F), dtype=np.float64)
    lib().orc_bias_geglu_fwd(_dt(x), rows, F, _ptr(x), _ptr(bias), _ptr(out))
    return out


def bias_geglu_bwd(g, x, bias=None, with_scale=False):
    """dx, or (dx, scale) with the per-element condition scale."""
    x = np.ascontiguousarray(x)
    g = np.ascontiguousarray(g)
    rows, two_f = x.shape
    F = two_f // 2
    assert g.shape == (rows, F) and g.dtype == x.dtype
    dx = np.empty((rows, 2 * F), dtype=np.float64)
    scale = np.empty((rows, 2 * F), dtype=np.float64) if with_scale else None
    lib().orc_bias_geglu_bwd(_dt(x), rows, F, _ptr(g), _ptr(x), _ptr(bias), _ptr(dx), _ptr(scale))
    return (dx, scale) if with_scale else dx


def bias_swiglu_fwd(x, bias=None, weight=None):
    x = np.ascontiguousarray(x)
    rows, two_f = x.shape
    F = two_f // 2
    if weight is not None:
        weight = np.ascontiguousarray(weight, dtype=np.float32).reshape(rows)
    out = np.empty((rows, F), dtype=np.float64)
    lib().orc_bias_swiglu_fwd(_dt(x), rows, F, _ptr(x), _ptr(bias), _ptr(weight), _ptr(out))
    return out


def bias_swiglu_bwd(g, x, bias=None, weight=None, with_scale=False):
    """Returns (dx, dweight, dweight_abs), plus the per-element condition
    scale of dx when with_scale; dweight and dweight_abs are None without a
    weight."""
    x = np.ascontiguousarray(x)
    g = np.ascontiguousarray(g)
    rows, two_f = x.shape
    F = two_f // 2
    assert g.shape == (rows, F) and g.dtype == x.dtype
    dx = np.empty((rows, 2 * F), dtype=np.float64)
    dw = dwa = None
    if weight is not None:
        weight = np.ascontiguousarray(weight, dtype=np.float32).reshape(rows)
        dw = np.empty(rows, dtype=np.float64)
        dwa = np.empty(rows, dtype=np.float64)
    scale = np.empty((rows, 2 * F), dtype=np.float64) if with_scale else None
    lib().orc_bias_swiglu_bwd(_dt(x), rows, F, _ptr(g), _ptr(x), _ptr(bias), _ptr(weight),
                              _ptr(dx), _ptr(dw), _ptr(dwa), _ptr(scale))
    return (dx, dw, dwa, scale) if with_scale else (dx, dw, dwa)


def bias_dropout_add_train(x, residual, bias=None, p=0.1, seed=0, offset=0, elem_base=0):
    """Returns (out, keep): out has x's dtype, keep is uint8 0/1."""
    x = np.ascontiguousarray(x)
    residual = np.ascontiguousarray(residual)
    rows, cols = x.shape
    assert residual.shape == x.shape
    out = np.empty_like(x)
    keep = np.empty((rows, cols), dtype=np.uint8)
    lib().orc_bias_dropout_add_train(_dt(x), _dt(residual), rows, cols, _ptr(x), _ptr(bias),
                                     _ptr(residual), float(p), seed, offset, elem_base,
                                     _ptr(out), _ptr(keep))
    return out, keep


def bias_dropout_add_inference(x, residual, bias=None):
    """In place on x (which must be a writable C-contiguous array); returns x."""
    assert x.flags["C_CONTIGUOUS"] and x.flags["WRITEABLE"]
    residual = np.ascontiguousarray(residual)
    rows, cols = x.shape
    lib().orc_bias_dropout_add_inference(_dt(x), _dt(residual), rows, cols, _ptr(x),
                                         _ptr(bias), _ptr(residual))
    return x


def bias_dropout_add_bwd(g, keep=None, p=0.1, seed=0, offset=0, elem_base=0, res_dtype=None):
    """(dx, dres): dx in g's dtype; dres in res_dtype ('bf16'/'f32', None = skip)."""
    g = np.ascontiguousarray(g)
    rows, cols = g.shape
    dx = np.empty_like(g)
    dres = None
    rdt = _dt(g)
    if res_dtype is not None:
        rdt = BF16 if res_dtype == "bf16" else F32
        dres = np.empty((rows, cols), dtype=np.uint16 if rdt == BF16 else np.float32)
    if keep is not None:
        keep = np.ascontiguousarray(keep, dtype=np.uint8)
    lib().orc_bias_dropout_add_bwd(_dt(g), rdt, rows, cols, _ptr(g), _ptr(keep), float(p), seed,
                                   offset, elem_base, _ptr(dx), _ptr(dres))
    return dx, dres


def column_sums(v, dtype):
    """(sum, abs_sum) over rows of v (float64 [rows, cols]) rounded to dtype
    ('bf16' or 'f32') first, as a stored gradient would be."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    s = np.empty(cols, dtype=np.float64)
    a = np.empty(cols, dtype=np.float64)
    lib().orc_column_sums(BF16 if dtype == "bf16" else F32, rows, cols, _ptr(v), _ptr(s), _ptr(a))
    return s, a


def weighted_squared_relu_fwd(x, weight):
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    w = np.ascontiguousarray(weight, dtype=np.float32).reshape(rows)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_weighted_squared_relu_fwd(_dt(x), rows, cols, _ptr(x), _ptr(w), _ptr(out))
    return out


def weighted_squared_relu_bwd(g, x, weight):
    """(dx, dweight, dweight_abs)."""
    x = np.ascontiguousarray(x)
    g = np.ascontiguousarray(g)
    rows, cols = x.shape
    w = np.ascontiguousarray(weight, dtype=np.float32).reshape(rows)
    dx = np.empty((rows, cols), dtype=np.float64)
    dw = np.empty(rows, dtype=np.float64)
    dwa = np.empty(rows, dtype=np.float64)
    lib().orc_weighted_squared_relu_bwd(_dt(x), rows, cols, _ptr(g), _ptr(x), _ptr(w), _ptr(dx), _ptr(dw), _ptr(dwa))
    return dx, dw, dwa


def scaled_masked_softmax_fwd(x, scale, mask=None, causal=False):
    """Softmax over the last dim of scale * x (+ additive mask) for x of 3 or
    4 dims ([attn_batches, sq, sk] or [b, np, sq, sk]); mask: 4 dims, each
    leading size 1 or x's.  Returns float64 of x's shape."""
    x = np.ascontiguousarray(x)
    shape = x.shape
    x4 = x.reshape((1,) * (4 - x.ndim) + shape)
    b, np_, sq, sk = x4.shape
    mb = mnp = msq = 1
    if mask is not None:
        mask = np.ascontiguousarray(mask)
        assert mask.dtype == x.dtype and mask.ndim == 4 and mask.shape[3] == sk
        mb, mnp, msq = mask.shape[:3]
        for m_, full in ((mb, b), (mnp, np_), (msq, sq)):
            assert m_ in (1, full)
    if causal:
        assert sq == sk
    y = np.empty(x4.shape, dtype=np.float64)
    lib().orc_scaled_masked_softmax_fwd(_dt(x), b, np_, sq, sk, _ptr(x), _ptr(mask), mb, mnp, msq,
                                        int(bool(causal)), float(scale), _ptr(y))
    return y.reshape(shape)


def scaled_softmax_bwd(dy, y, scale, causal=False, with_scale=False):
    """dx (float64, y's shape) from the upstream gradient and the forward's
    rounded outputs (both of y's dtype); with_scale also returns the
    condition scale of each element."""
    dy = np.ascontiguousarray(dy)
    y = np.ascontiguousarray(y)
    assert dy.dtype == y.dtype and dy.shape == y.shape
    sk = y.shape[-1]
    rows = y.size // sk if sk else 0
    if causal:
        assert y.ndim >= 2 and y.shape[-2] == sk
    dx = np.empty(y.shape, dtype=np.float64)
    sc = np.empty(y.shape, dtype=np.float64)
    lib().orc_scaled_softmax_bwd(_dt(y), rows, sk, _ptr(dy), _ptr(y), int(bool(causal)), float(scale),
                                 _ptr(dx), _ptr(sc))
    return (dx, sc) if with_scale else dx
