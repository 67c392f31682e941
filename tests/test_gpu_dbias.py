"""Fused bias gradients (NEXT row f2): dbias = column sums of the stored
backward gradient.  Checked (1) bit for bit against a float32 replay of the
documented two-stage summation order (tests/dbias_order.py), with the partial
count J read off a NaN-filled workspace, so a dropped, doubled or misplaced
term fails; (2) against the float64 column sums of the stored gradient within
the error bound of that order (each term passes through about rows/J + J/256
+ 13 fp32 additions) plus one final rounding; (3) against the oracle's column
sums with the bound the elementwise parity implies; (4) bitwise run to run;
and through the workspace protocol.  Full-size cases cover the layer shapes
the benchmark times."""
import ctypes as C

import numpy as np
import pytest
import torch

import dbias_order as DBO
import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bf16_ulp, bits, check, f32_ulp, to_f64

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


class NanWorkspace:
    """An allocator for the binding's workspace hook: hands out a workspace
    whose words are all NaN and keeps it for inspection."""

    def __init__(self):
        self.ws = None

    def __call__(self, nbytes):
        self.ws = DBO.nan_workspace(nbytes, DEV)
        return self.ws


def check_dbias(dbias, stored, ws, ref_rows=None, dtype_name=None):
    """(1) bitwise against the replay of the summation order; (2) against the
    float64 sums of the stored gradient within that order's bound; (3)
    optionally against the oracle's exact gradient rows ref_rows (float64
    [rows, W]).  Returns J."""
    Wd = stored.shape[-1]
    J = DBO.partials_written(ws.ws, Wd)
    st32 = stored.detach().float().cpu().numpy().reshape(-1, Wd)
    rows = st32.shape[0]
    rep = torch.from_numpy(DBO.replay(st32, J)).to(dbias.dtype)
    assert np.array_equal(bits(rep), bits(dbias)), \
        f"dbias differs from the replayed order at {np.flatnonzero(bits(rep) != bits(dbias))[:5]} (J={J})"
    got = to_f64(dbias)
    exact, mag = DBO.column_sums(st32)
    tol = DBO.tolerance(got, exact, mag, rows, J, dbias.dtype == BF16)
    err = np.abs(got - exact)
    assert np.all(err <= tol), float(np.max(err / tol))
    if ref_rows is not None:
        rs, _ = O.column_sums(ref_rows, dtype_name)
        # every stored element is within one ulp of its reference (bf16) or
        # within 1e-6 / 2 ulp (fp32): the sums differ by at most those errors
        elem = (bf16_ulp(ref_rows) if dtype_name == "bf16" else np.maximum(1e-6, 2 * f32_ulp(ref_rows)))
        assert np.all(np.abs(got - rs) <= tol + elem.sum(axis=0))
    return J


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(1, 8), (3, 24), (64, 1024), (33, 4104), (200, 4096), (9, 4099)])
def test_gelu_dbias(dtype, shape):
    rows, cols = shape
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=rows + cols)
    ws = NanWorkspace()
    dy, db = mfx.mfx_bias_gelu_bwd_dbias(on(g), on(b), on(y), workspace=ws)
    dy_plain = mfx.mfx_bias_gelu_bwd(on(g), on(b), on(y))
    torch.cuda.synchronize()
    assert np.array_equal(bits(dy), bits(dy_plain))  # the fused call's dy is the plain call's
    ref = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b))
    check_dbias(db, dy, ws, ref, "bf16" if dtype == BF16 else "f32")


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(3, 8), (7, 1024), (13, 2400), (3, 4099), (40, 14336)])
def test_glu_dbias(kind, dtype, shape):
    rows, F = shape
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=rows * 3 + F, with_weight=kind == "swiglu_w")
    ws = NanWorkspace()
    if kind == "geglu":
        dx, db = mfx.mfx_bias_geglu_bwd_dbias(on(g), on(x), on(b), workspace=ws)
        dx_plain = mfx.mfx_bias_geglu_bwd(on(g), on(x), on(b))
        ref = O.bias_geglu_bwd(W.to_oracle(g), W.to_oracle(x), W.to_oracle(b))
    else:
        dx, dw, db = mfx.mfx_bias_swiglu_bwd_dbias(on(g), on(x), on(b), on(w), workspace=ws)
        dx_plain, _ = mfx.mfx_bias_swiglu_bwd(on(g), on(x), on(b), on(w))
        ref = O.bias_swiglu_bwd(W.to_oracle(g), W.to_oracle(x), W.to_oracle(b), W.to_oracle(w))[0]
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx), bits(dx_plain))
    check_dbias(db, dx, ws, ref, "bf16" if dtype == BF16 else "f32")


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (F32, F32), (BF16, BF16)])
@pytest.mark.parametrize("shape", [(2, 8), (16, 4096), (5, 24), (3, 4099), (64, 1032)])
@pytest.mark.parametrize("regen", [False, True])
def test_dropout_dbias(xdt, rdt, shape, regen):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + cols)
    g = W.normal((rows, cols), xdt, 3)
    _, keep = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), 0.25, 7, 1)
    ws = NanWorkspace()
    dx, dres, db = mfx.mfx_bias_dropout_add_bwd_dbias(on(g), None if regen else keep, 0.25, 7, 1,
                                                      residual_dtype=rdt, workspace=ws)
    dx_plain, _ = mfx.mfx_bias_dropout_add_bwd(on(g), keep, 0.25)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx), bits(dx_plain))
    check_dbias(db, dx, ws)


@pytest.mark.parametrize("op", ["gelu", "dropout"])
def test_dbias_many_partials(op):
    """Hundreds of partial rows per column (a full grid over narrow rows), so
    the finish kernel runs its eight-wide main loop as well as its tail."""
    ws = [NanWorkspace(), NanWorkspace()]
    if op == "gelu":
        y, b, g = W.gelu_inputs(8192, 1024, BF16, seed=12)
        runs = [mfx.mfx_bias_gelu_bwd_dbias(on(g), on(b), on(y), workspace=w) for w in ws]
        stored, db = runs[0]
        dbs = [r[1] for r in runs]
    else:
        g = W.normal((8192, 1024), BF16, 13)
        runs = [mfx.mfx_bias_dropout_add_bwd_dbias(on(g), None, 0.1, 1234, 0, residual_dtype=F32, workspace=w)
                for w in ws]
        stored, _, db = runs[0]
        dbs = [r[2] for r in runs]
    torch.cuda.synchronize()
    J = check_dbias(db, stored, ws[0])
    assert J > 8 * DBO.FINISH_WARPS
    assert np.array_equal(bits(dbs[0]), bits(dbs[1]))


def test_dbias_is_bitwise_reproducible_and_paths_agree():
    y, b, g = W.gelu_inputs(512, 4096, BF16, seed=9)
    yd, bd, gd = on(y), on(b), on(g)
    runs = [mfx.mfx_bias_gelu_bwd_dbias(gd, bd, yd)[1].clone() for _ in range(3)]
    ws = NanWorkspace()
    _, db_m = mfx.mfx_bias_gelu_bwd_dbias(misaligned(g), misaligned(b), misaligned(y),
                                          dy=misaligned(torch.zeros_like(y)), workspace=ws)
    dy = mfx.mfx_bias_gelu_bwd(gd, bd, yd)
    torch.cuda.synchronize()
    for r in runs[1:]:
        assert np.array_equal(bits(runs[0]), bits(r))
    check_dbias(db_m, dy, ws)      # the fallback (generic + column partials) is right too
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
    ws = DBO.nan_workspace(need + 32, DEV)
    small = C.c_size_t(need - 16)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr(), C.byref(small), None) == 8
    odd = C.c_size_t(need)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr() + 4, C.byref(odd), None) == 8
    torch.cuda.synchronize()
    assert torch.all(ws == 0xFF).item()        # refused calls launch nothing
    ok = C.c_size_t(need)
    assert L.mfx_bias_gelu_bwd_dbias(1, 64, 1024, gd.data_ptr(), bd.data_ptr(), yd.data_ptr(), dy.data_ptr(),
                                     db.data_ptr(), ws.data_ptr(), C.byref(ok), None) == 0
    # an empty batch has a zero bias gradient
    db2 = torch.full((1024,), 7.0, dtype=BF16, device=DEV)
    e = torch.empty(0, 1024, dtype=BF16, device=DEV)
    _, db2 = mfx.mfx_bias_gelu_bwd_dbias(e, bd, e, dbias=db2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(db2).item() == 0
    holder = NanWorkspace()
    holder.ws = ws
    J = check_dbias(db, dy, holder)
    assert J * 1024 * 4 <= need                  # the query covered what the call wrote


# ---------------------------------------------------------------------------
# Full size: the layer shapes the benchmark times, 16384 rows.
# ---------------------------------------------------------------------------
def same_bits(a, b):
    """Bitwise equality of two CUDA tensors of one dtype, on the device."""
    iv = torch.int16 if a.dtype == BF16 else torch.int32
    return bool(torch.equal(a.contiguous().view(iv), b.contiguous().view(iv)))


def check_full(db, stored, ws, again):
    """check_dbias plus: run-to-run bits, and a planted dropped row (on the
    CPU, in the replayed order) fails both the bitwise and the bound check."""
    J = check_dbias(db, stored, ws)
    assert same_bits(db, again)
    Wd = stored.shape[-1]
    st32 = stored.float().cpu().numpy().reshape(-1, Wd)
    dropped = st32.copy()
    dropped[st32.shape[0] // 2] = 0.0
    rep = torch.from_numpy(DBO.replay(dropped, J)).to(db.dtype)
    assert not np.array_equal(bits(rep), bits(db))
    exact, mag = DBO.column_sums(st32)
    got = to_f64(rep)
    tol = DBO.tolerance(got, exact, mag, st32.shape[0], J, db.dtype == BF16)
    assert np.any(np.abs(got - exact) > tol)
    return J


@pytest.mark.parametrize("cols", [16384, 4099])
def test_gelu_dbias_bf16_16384_rows(cols):
    """16384 x 16384 (the pipelined kernel's partials) and 16384 x 4099
    (generic backward + the column-partial pass)."""
    y, b, g = W.gelu_inputs(16384, cols, BF16, seed=21, device=DEV)
    ws = NanWorkspace()
    dy, db = mfx.mfx_bias_gelu_bwd_dbias(g, b, y, workspace=ws)
    dy_plain = mfx.mfx_bias_gelu_bwd(g, b, y)
    again = mfx.mfx_bias_gelu_bwd_dbias(g, b, y)[1]
    torch.cuda.synchronize()
    assert same_bits(dy, dy_plain)
    check_full(db, dy, ws, again)
    # the stored gradient itself, on sampled rows, against the oracle
    rs = torch.tensor([0, 5, 8191, 16383], device=DEV)
    ref, scale = O.bias_gelu_bwd(W.to_oracle(g[rs]), W.to_oracle(y[rs]), W.to_oracle(b), with_scale=True)
    check(dy[rs], ref, "dy rows", scale)
    assert mfx.mfx_device_error() == 0


def test_geglu_dbias_bf16_16384x28672():
    x, b, g, _ = W.glu_inputs(16384, 14336, BF16, seed=22, device=DEV)
    ws = NanWorkspace()
    dx, db = mfx.mfx_bias_geglu_bwd_dbias(g, x, b, workspace=ws)
    dx_plain = mfx.mfx_bias_geglu_bwd(g, x, b)
    again = mfx.mfx_bias_geglu_bwd_dbias(g, x, b)[1]
    torch.cuda.synchronize()
    assert same_bits(dx, dx_plain)
    check_full(db, dx, ws, again)
    assert mfx.mfx_device_error() == 0


@pytest.mark.parametrize("regen", [False, True])
def test_dropout_dbias_bf16_16384x4096(regen):
    """The residual-add shape [4096 x 4] x 4096, fp32 residual, p = 0.1, seed
    1234: the gradient through the dropout mask, read or regenerated."""
    x, b, r = W.dropout_inputs(16384, 4096, BF16, F32, seed=23, device=DEV)
    g = W.normal((16384, 4096), BF16, 24, device=DEV)
    _, keep = mfx.mfx_bias_dropout_add_train(x, b, r, 0.1, 1234, 0)
    ws = NanWorkspace()
    mask = None if regen else keep
    dx, dres, db = mfx.mfx_bias_dropout_add_bwd_dbias(g, mask, 0.1, 1234, 0, residual_dtype=F32, workspace=ws)
    dx_plain, _ = mfx.mfx_bias_dropout_add_bwd(g, keep, 0.1)
    again = mfx.mfx_bias_dropout_add_bwd_dbias(g, mask, 0.1, 1234, 0, residual_dtype=F32)[2]
    torch.cuda.synchronize()
    assert same_bits(dx, dx_plain)
    assert torch.equal(dres, g.float())
    check_full(db, dx, ws, again)
    assert mfx.mfx_device_error() == 0
