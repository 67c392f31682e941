"""GLU at any F (from 64 columns) and any alignment.

Units are 8 consecutive elements of the forward output's (backward: g's)
flat grid, aligned to its 16-byte boundaries; the a and b runs, and the
backward's outputs, sit at any alignment and go through aligned vectors
(realigned loads, stores assembled across the warp); units that straddle a
row boundary are done element by element in a last pass.  Checked against
the oracle at odd widths and widths around 2048, with each tensor at its own
element offset; in-place backward; and bit for bit against the aligned
fixed-column path where one exists (F % 8 == 0), including the weighted
SwiGLU's row-sum weight gradient."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bits, check, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def at_offset(t, k):
    if t is None:
        return None
    t = t.to(DEV)
    buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[k:k + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def run(kind, x, b, g, w, offs):
    """fwd, dx, dweight with x, b, g, out, dx at element offsets offs."""
    ox, ob, og, oo, od = offs
    xk, bk, gk = at_offset(x, ox), at_offset(b, ob), at_offset(g, og)
    rows, two_f = x.shape
    out = at_offset(torch.zeros(rows, two_f // 2, dtype=x.dtype), oo)
    dx = at_offset(torch.zeros_like(x), od)
    wd = None if w is None else w.to(DEV)
    if kind == "geglu":
        mfx.mfx_bias_geglu_fwd(xk, bk, out=out)
        mfx.mfx_bias_geglu_bwd(gk, xk, bk, dx=dx)
        return out, dx, None
    mfx.mfx_bias_swiglu_fwd(xk, bk, wd, out=out)
    _, dw = mfx.mfx_bias_swiglu_bwd(gk, xk, bk, wd, dx=dx)
    return out, dx, dw


def oracle(kind, x, b, g, w):
    xo, bo, go, wo = W.to_oracle(x), W.to_oracle(b), W.to_oracle(g), W.to_oracle(w)
    if kind == "geglu":
        dx, sc = O.bias_geglu_bwd(go, xo, bo, with_scale=True)
        return O.bias_geglu_fwd(xo, bo), dx, sc, None, None
    dx, dw, dwa, sc = O.bias_swiglu_bwd(go, xo, bo, wo, with_scale=True)
    return O.bias_swiglu_fwd(xo, bo, wo), dx, sc, dw, dwa


OFFSETS = [(0, 0, 0, 0, 0), (1, 0, 0, 0, 0), (0, 3, 5, 1, 7), (3, 1, 2, 5, 3), (7, 7, 7, 7, 7)]


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(3, 64), (5, 65), (4, 1023), (3, 2047), (2, 2049), (3, 4099), (2, 6001),
                                   (9, 100)])
def test_glu_any_width_against_oracle(kind, dtype, shape):
    rows, F = shape
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=rows * 31 + F, with_weight=kind == "swiglu_w")
    ref_f, ref_dx, sc, ref_dw, ref_dwa = oracle(kind, x, b, g, w)
    first = None
    for offs in OFFSETS if dtype == BF16 else [o for o in OFFSETS if max(o) < 4] + [(1, 2, 3, 0, 1)]:
        f, dx, dw = run(kind, x, b, g, w, offs)
        torch.cuda.synchronize()
        check(f, ref_f, f"{kind} fwd {offs}")
        check(dx, ref_dx, f"{kind} bwd {offs}", sc)
        if dw is not None:
            err = np.abs(to_f64(dw) - ref_dw)
            assert np.all(err <= 1e-5 * ref_dwa + 1e-30)
        got = (bits(f), bits(dx), None if dw is None else bits(dw))
        if first is None:
            first = got
        else:                                    # every placement gives the same bits
            assert np.array_equal(got[0], first[0]) and np.array_equal(got[1], first[1])
            if dw is not None:
                assert np.array_equal(got[2], first[2])
    assert mfx.mfx_device_error() == 0


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", [BF16, F32])
def test_glu_misaligned_matches_aligned_path_bitwise(kind, dtype):
    """F % 8 == 0: aligned buffers take the fixed-column path, buffers one
    element off the realigning one; outputs and weight gradient agree."""
    rows, F = 7, 4104
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=5, with_weight=kind == "swiglu_w")
    fa, dxa, dwa = run(kind, x, b, g, w, (0, 0, 0, 0, 0))
    fm, dxm, dwm = run(kind, x, b, g, w, (1, 1, 1, 1, 1))
    torch.cuda.synchronize()
    assert np.array_equal(bits(fa), bits(fm)) and np.array_equal(bits(dxa), bits(dxm))
    if dwa is not None:
        assert np.array_equal(bits(dwa), bits(dwm))


@pytest.mark.parametrize("kind", ["geglu", "swiglu_w"])
def test_glu_any_width_in_place_backward(kind):
    rows, F = 6, 4099
    x, b, g, w = W.glu_inputs(rows, F, BF16, seed=8, with_weight=kind == "swiglu_w")
    _, ref_dx, sc, _, _ = oracle(kind, x, b, g, w)
    xk = at_offset(x, 3)
    if kind == "geglu":
        mfx.mfx_bias_geglu_bwd(at_offset(g, 1), xk, at_offset(b, 2), dx=xk)
    else:
        mfx.mfx_bias_swiglu_bwd(at_offset(g, 1), xk, at_offset(b, 2), w.to(DEV), dx=xk)
    torch.cuda.synchronize()
    check(xk, ref_dx, f"{kind} in-place bwd", sc)


def test_glu_odd_layer_width_sampled_rows():
    """16384 x (2 x 4099) bf16 (the sweep's odd width), sampled rows."""
    rows, F = 16384, 4099
    x, b, g, _ = W.glu_inputs(rows, F, BF16, seed=12, device=DEV)
    f = mfx.mfx_bias_swiglu_fwd(x, b)
    dx, _ = mfx.mfx_bias_swiglu_bwd(g, x, b)
    torch.cuda.synchronize()
    rs = torch.tensor([0, 1, 4097, 8191, 16383], device=DEV)
    xo, bo, go = W.to_oracle(x[rs]), W.to_oracle(b), W.to_oracle(g[rs])
    check(f[rs], O.bias_swiglu_fwd(xo, bo), "swiglu fwd rows")
    ref, _, _, sc = O.bias_swiglu_bwd(go, xo, bo, None, with_scale=True)
    check(dx[rs], ref, "swiglu bwd rows", sc)


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("F,rows", [(64, 1237), (192, 1237), (1024, 1237), (1032, 1237), (2048, 1237), (8, 301),
                                    (16, 1), (1024, 1)])
def test_weighted_short_rows_packed_stage(dtype, F, rows):
    """Rows of at most 256 units share a stage (64 down to 2 rows of the
    block per stage; F = 1032 puts a row slot across both units of a
    consumer).  Row counts leave the last stage of each block ragged.  dx
    and dweight equal the bits of the realigning path (pointers one element
    off), and dweight is within the summation bound of the oracle's."""
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=F + 7, with_weight=True)
    fa, dxa, dwa = run("swiglu_w", x, b, g, w, (0, 0, 0, 0, 0))
    fm, dxm, dwm = run("swiglu_w", x, b, g, w, (1, 1, 1, 1, 1))
    torch.cuda.synchronize()
    assert np.array_equal(bits(dxa), bits(dxm)) and np.array_equal(bits(dwa), bits(dwm))
    _, ref_dx, sc, ref_dw, ref_dwa = oracle("swiglu_w", x, b, g, w)
    check(dxa, ref_dx, "dx", sc)
    assert np.all(np.abs(to_f64(dwa) - ref_dw) <= 1e-5 * ref_dwa + 1e-30)
    assert mfx.mfx_device_error() == 0


@pytest.mark.parametrize("kind", ["geglu", "swiglu_w"])
def test_glu_misaligned_layer_width_whole_tensor_bitwise(kind):
    """2048 x (2 x 14336) bf16 with every pointer one element off 16 bytes
    (the realigning ring; its first and last rows meet the clipped vectors
    at the ends of x and g) against the aligned pipeline: the whole of the
    forward output, dx and dweight bit for bit."""
    rows, F = 2048, 14336
    x, b, g, w = W.glu_inputs(rows, F, BF16, seed=23, with_weight=kind == "swiglu_w")
    fa, dxa, dwa = run(kind, x, b, g, w, (0, 0, 0, 0, 0))
    fm, dxm, dwm = run(kind, x, b, g, w, (1, 1, 1, 1, 1))
    torch.cuda.synchronize()
    assert torch.equal(fa.view(torch.int16), fm.view(torch.int16))
    assert torch.equal(dxa.view(torch.int16), dxm.view(torch.int16))
    if dwa is not None:
        assert torch.equal(dwa.view(torch.int32), dwm.view(torch.int32))
    assert mfx.mfx_device_error() == 0
