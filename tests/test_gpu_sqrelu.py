"""Parity of the weighted squared ReLU kernels (through the C ABI) with the
CPU oracle: ragged and multi-chunk shapes, the pipelined and generic paths,
in-place and misaligned buffers, extreme values and the reproducibility of
the weight gradient.  Tolerances: tests/parity.py (bf16: 1 ulp; fp32: 1e-6
or 2 ulps; dweight: 1e-5 of the row's sum of |terms|)."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import F32_OVERFLOW, bits, check, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16]
BF16 = torch.bfloat16

# (1, 1) .. (5, 16384): ragged widths take the generic kernels; widths that
# are multiples of 8 take the pipelined ones, (3, 2056) and (2, 16384) with
# several 256-unit chunks per row in the backward, (300, 24) with many rows
# per block.
SHAPES = [(1, 1), (1, 7), (2, 9), (3, 4099), (17, 24), (300, 24), (64, 1024), (3, 2056), (33, 4104),
          (5, 16384), (2, 16384), (3, 14336), (2, 16392), (2, 32768)]


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
    assert v.data_ptr() % 16 != 0 and v.is_contiguous()
    return v


def _ref(x, g, w):
    xo, go, wo = W.to_oracle(x), W.to_oracle(g), W.to_oracle(w)
    f = O.weighted_squared_relu_fwd(xo, wo)
    dx, dw, dwa = O.weighted_squared_relu_bwd(go, xo, wo)
    return f, dx, dw, dwa


def check_dweight(dw, ref, ref_abs, what):
    err = np.abs(to_f64(dw) - ref)
    assert np.all(err <= 1e-5 * ref_abs + 1e-30), f"{what}: max rel-to-abs-sum {np.max(err / (ref_abs + 1e-30)):.3e}"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
def test_weighted_squared_relu(dtype, shape):
    rows, cols = shape
    x, g, w = W.sqrelu_inputs(rows, cols, dtype, seed=rows * 7 + cols)
    ref_f, ref_dx, ref_dw, ref_dwa = _ref(x, g, w)
    xd, gd, wd = on(x), on(g), on(w)
    f = mfx.mfx_weighted_squared_relu_fwd(xd, wd)
    dx, dw = mfx.mfx_weighted_squared_relu_bwd(gd, xd, wd)
    torch.cuda.synchronize()
    check(f, ref_f, f"sqrelu fwd {dtype} {shape}")
    check(dx, ref_dx, f"sqrelu bwd {dtype} {shape}")
    check_dweight(dw, ref_dw, ref_dwa, f"sqrelu dweight {dtype} {shape}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_misaligned_and_in_place_match_aligned(dtype):
    rows, cols = 6, 2056
    x, g, w = W.sqrelu_inputs(rows, cols, dtype, seed=5)
    xd, gd, wd = on(x), on(g), on(w)
    f = mfx.mfx_weighted_squared_relu_fwd(xd, wd)
    dx, dw = mfx.mfx_weighted_squared_relu_bwd(gd, xd, wd)
    fm = mfx.mfx_weighted_squared_relu_fwd(misaligned(x), wd, out=misaligned(torch.zeros_like(x)))
    dxm, dwm = mfx.mfx_weighted_squared_relu_bwd(misaligned(g), misaligned(x), wd,
                                                 dx=misaligned(torch.zeros_like(x)))
    xi = xd.clone()
    fi = mfx.mfx_weighted_squared_relu_fwd(xi, wd, out=xi)
    xi2, gi = xd.clone(), gd.clone()
    dxi, dwi = mfx.mfx_weighted_squared_relu_bwd(gi, xi2, wd, dx=xi2)
    dxg, dwg = mfx.mfx_weighted_squared_relu_bwd(gi.clone(), xd, wd, dx=None)
    torch.cuda.synchronize()
    assert np.array_equal(bits(f), bits(fm)) and np.array_equal(bits(f), bits(fi))
    assert np.array_equal(bits(dx), bits(dxm)) and np.array_equal(bits(dx), bits(dxi))
    # the generic backward sums the row in another order: compare within the
    # weight-gradient bound, and its dx bit for bit
    _, _, ref_dw, ref_dwa = _ref(x, g, w)
    check_dweight(dwm, ref_dw, ref_dwa, "misaligned dweight")
    assert np.array_equal(bits(dw), bits(dwi)) and np.array_equal(bits(dw), bits(dwg))


def test_dweight_is_deterministic():
    x, g, w = W.sqrelu_inputs(300, 4104, BF16, seed=4)
    xd, gd, wd = on(x), on(g), on(w)
    outs = [mfx.mfx_weighted_squared_relu_bwd(gd, xd, wd)[1].clone() for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert np.array_equal(bits(outs[0]), bits(o))


@pytest.mark.parametrize("dtype", DTYPES)
def test_extreme_values(dtype):
    """Overflow to inf where the exact result overflows, zero weights, NaN
    inputs (relu(NaN) = 0 in the oracle's comparison form too) and the
    largest finite inputs, whose gradient 2 w x stays finite for w <= 1/2."""
    a = torch.cat([torch.linspace(-40, 40, 4000),
                   torch.tensor([1e20, -1e20, 0.0, -0.0, 3e38, -3e38, 1e19, 1.8e19, float("nan"), 1e-30,
                                 2.0, -2.0, 0.5, 1e-20, 1e-38, 65504.0])])
    cols = a.numel()
    assert cols % 8 == 0  # the pipelined kernels take these rows
    x = torch.stack([a, a, a, -a]).to(dtype)
    g = torch.ones(4, cols).to(dtype)
    w = torch.tensor([0.5, 0.0, 1e-30, 0.25], dtype=torch.float32)
    ref_f, ref_dx, ref_dw, ref_dwa = _ref(x, g, w)
    f = mfx.mfx_weighted_squared_relu_fwd(on(x), on(w))
    dx, dw = mfx.mfx_weighted_squared_relu_bwd(on(g), on(x), on(w))
    torch.cuda.synchronize()
    check(f, ref_f, f"sqrelu fwd extremes {dtype}")
    check(dx, ref_dx, f"sqrelu bwd extremes {dtype}")
    got = to_f64(dw)
    sat = np.abs(ref_dw) >= F32_OVERFLOW
    assert np.all(np.isinf(got[sat]) & (got[sat] > 0))
    assert np.all(np.abs(got[~sat] - ref_dw[~sat]) <= 1e-5 * ref_dwa[~sat] + 1e-30)


def test_empty_and_argument_errors():
    x = torch.zeros(0, 64, dtype=BF16, device=DEV)
    w = torch.zeros(0, dtype=torch.float32, device=DEV)
    assert mfx.mfx_weighted_squared_relu_fwd(x, w).shape == (0, 64)
    L = mfx.lib()
    assert L.mfx_weighted_squared_relu_fwd(1, 4, 8, None, None, None, None) == 1  # NULL
    assert L.mfx_weighted_squared_relu_fwd(9, 4, 8, None, None, None, None) == 3  # dtype
    assert L.mfx_weighted_squared_relu_bwd(1, -1, 8, None, None, None, None, None, None) == 2  # shape
    xs = torch.ones(4, 8, dtype=BF16, device=DEV)
    ws = torch.ones(4, dtype=torch.float32, device=DEV)
    dw = torch.empty(4, dtype=torch.float32, device=DEV)
    # dweight inside dx's buffer
    assert L.mfx_weighted_squared_relu_bwd(1, 4, 8, xs.data_ptr(), xs.data_ptr(), ws.data_ptr(),
                                           xs.data_ptr(), xs.data_ptr() + 16, None) == 5
    assert L.mfx_weighted_squared_relu_bwd(1, 4, 8, xs.data_ptr(), xs.data_ptr(), ws.data_ptr(),
                                           xs.data_ptr(), dw.data_ptr(), None) == 0
    with pytest.raises(ValueError):
        mfx.mfx_weighted_squared_relu_fwd(xs, torch.ones(3, dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert mfx.mfx_device_error() == 0
