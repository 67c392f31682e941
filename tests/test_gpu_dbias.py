"""Fused bias gradients (NEXT row f2): dbias = column sums of the stored
backward gradient.  Checked (1) tightly against the float64 column sums of
the gradient the GPU stored (fp32 summation error + one final rounding),
(2) against the oracle's column sums with the bound the elementwise parity
implies (each stored element is within its own tolerance), (3) bitwise run
to run, and through the workspace protocol."""
import ctypes as C

import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bf16_ulp, bits, f32_ulp, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def on(t):
    return None if t is None else t.to(DEV)


def misaligned(t):
    buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def check_dbias(dbias, stored, ref_rows=None, dtype_name=None):
    """(1) against the sums of the stored gradient; (2) optionally against the
    oracle's exact gradient rows ref_rows (float64 [rows, W])."""
    st = to_f64(stored)
    got = to_f64(dbias)
    s = st.sum(axis=0)
    a = np.abs(st).sum(axis=0)
    ulp = bf16_ulp if dbias.dtype == BF16 else f32_ulp
    rows = st.shape[0]
    tol = ulp(s) + rows * 2.0 ** -23 * a
    assert np.all(np.abs(got - s) <= tol), float(np.max(np.abs(got - s) / tol))
    if ref_rows is not None:
        rs, ra = O.column_sums(ref_rows, dtype_name)
        # every stored element is within one ulp of its reference (bf16) or
        # within 1e-6 / 2 ulp (fp32): the sums differ by at most those errors
        elem = (bf16_ulp(ref_rows) if dtype_name == "bf16" else np.maximum(1e-6, 2 * f32_ulp(ref_rows)))
        tol2 = ulp(rs) + elem.sum(axis=0) + rows * 2.0 ** -23 * ra
        assert np.all(np.abs(got - rs) <= tol2)


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(1, 8), (3, 24), (64, 1024), (33, 4104), (200, 4096), (9, 4099)])
def test_gelu_dbias(dtype, shape):
    rows, cols = shape
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=rows + cols)
    dy, db = mfx.mfx_bias_gelu_bwd_dbias(on(g), on(b), on(y))
    dy_plain = mfx.mfx_bias_gelu_bwd(on(g), on(b), on(y))
    torch.cuda.synchronize()
    assert np.array_equal(bits(dy), bits(dy_plain))  # the fused call's dy is the plain call's
    ref = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b))
    check_dbias(db, dy, ref, "bf16" if dtype == BF16 else "f32")


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(3, 8), (7, 1024), (13, 2400), (3, 4099), (40, 14336)])
def test_glu_dbias(kind, dtype, shape):
    rows, F = shape
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=rows * 3 + F, with_weight=kind == "swiglu_w")
    if kind == "geglu":
        dx, db = mfx.mfx_bias_geglu_bwd_dbias(on(g), on(x), on(b))
        dx_plain = mfx.mfx_bias_geglu_bwd(on(g), on(x), on(b))
        ref = O.bias_geglu_bwd(W.to_oracle(g), W.to_oracle(x), W.to_oracle(b))
    else:
        dx, dw, db = mfx.mfx_bias_swiglu_bwd_dbias(on(g), on(x), on(b), on(w))
        dx_plain, _ = mfx.mfx_bias_swiglu_bwd(on(g), on(x), on(b), on(w))
        ref = O.bias_swiglu_bwd(W.to_oracle(g), W.to_oracle(x), W.to_oracle(b), W.to_oracle(w))[0]
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx), bits(dx_plain))
    check_dbias(db, dx, ref, "bf16" if dtype == BF16 else "f32")


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (F32, F32), (BF16, BF16)])
@pytest.mark.parametrize("shape", [(2, 8), (16, 4096), (5, 24), (3, 4099), (64, 1032)])
@pytest.mark.parametrize("regen", [False, True])
def test_dropout_dbias(xdt, rdt, shape, regen):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + cols)
    g = W.normal((rows, cols), xdt, 3)
    _, keep = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), 0.25, 7, 1)
    dx, dres, db = mfx.mfx_bias_dropout_add_bwd_dbias(on(g), None if regen else keep, 0.25, 7, 1,
                                                      residual_dtype=rdt)
    dx_plain, _ = mfx.mfx_bias_dropout_add_bwd(on(g), keep, 0.25)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx), bits(dx_plain))
    check_dbias(db, dx)


@pytest.mark.parametrize("op", ["gelu", "dropout"])
def test_dbias_many_partials(op):
    """Hundreds of partial rows per column (a full grid over narrow rows), so
    the finish kernel runs its eight-wide main loop as well as its tail."""
    if op == "gelu":
        y, b, g = W.gelu_inputs(8192, 1024, BF16, seed=12)
        dy, db = mfx.mfx_bias_gelu_bwd_dbias(on(g), on(b), on(y))
        stored = dy
    else:
        g = W.normal((4096, 4096), BF16, 13)
        stored, _, db = mfx.mfx_bias_dropout_add_bwd_dbias(on(g), None, 0.1, 1234, 0, residual_dtype=F32)
    runs = [db.clone()]
    if op == "gelu":
        runs.append(mfx.mfx_bias_gelu_bwd_dbias(on(g), on(b), on(y))[1])
    else:
        runs.append(mfx.mfx_bias_dropout_add_bwd_dbias(on(g), None, 0.1, 1234, 0, residual_dtype=F32)[2])
    torch.cuda.synchronize()
    check_dbias(db, stored)
    assert np.array_equal(bits(runs[0]), bits(runs[1]))


def test_dbias_is_bitwise_reproducible_and_paths_agree():
    y, b, g = W.gelu_inputs(512, 4096, BF16, seed=9)
    yd, bd, gd = on(y), on(b), on(g)
    runs = [mfx.mfx_bias_gelu_bwd_dbias(gd, bd, yd)[1].clone() for _ in range(3)]
    _, db_m = mfx.mfx_bias_gelu_bwd_dbias(misaligned(g), misaligned(b), misaligned(y),
                                          dy=misaligned(torch.zeros_like(y)))
    dy = mfx.mfx_bias_gelu_bwd(gd, bd, yd)
    torch.cuda.synchronize()
    for r in runs[1:]:
        assert np.array_equal(bits(runs[0]), bits(r))
    check_dbias(db_m, dy)          # the fallback (generic + column partials) is right too
    assert mfx.mfx_device_error() == 0


def test_workspace_protocol():
    L = mfx.lib()
    y, b, g = W.gelu_inputs(64, 1024, BF16, seed=2)
    yd, bd, gd = on(y), on(b), on(g)
    dy = torch.empty_like(yd)
    db = torch.empty(1024, dtype=BF16, device=DEV)
    size = C.c_size_t(0)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), None, C.byref(size), None) == 0
    need = size.value
    assert need >= 1024 * 4 and need % 16 == 0
    ws = torch.empty(need + 32, dtype=torch.uint8, device=DEV)
    small = C.c_size_t(need - 16)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr(), C.byref(small), None) == 8
    odd = C.c_size_t(need)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr() + 4, C.byref(odd), None) == 8
    ok = C.c_size_t(need)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr(), C.byref(ok), None) == 0
    # an empty batch has a zero bias gradient
    db2 = torch.full((1024,), 7.0, dtype=BF16, device=DEV)
    e = torch.empty(0, 1024, dtype=BF16, device=DEV)
    _, db2 = mfx.mfx_bias_gelu_bwd_dbias(e, bd, e, dbias=db2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(db2).item() == 0
    check_dbias(db, dy)
