"""Pins of the scale-mask-softmax oracle (fusions page §6.2-§6.4 of the web
page "Megatron-LM operator fusion walkthrough", www.wmrh.cn/news/51426)
against things other than itself: the page's worked causal example, the
closed form of the causal softmax of zeros, scipy's and torch's softmax,
numpy broadcasting of the mask, central differences of the forward, and the
identities a softmax Jacobian satisfies.  Each docstring names the mistakes
the test is there to catch."""
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

import oracle as O
from elementwise_epilogues_transformer_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_causal_zero.txt")


def _x(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def _dyadic(shape, seed):
    return (np.round(np.random.default_rng(seed).standard_normal(shape) * 64) / 64).astype(np.float32)


def test_page_causal_zero_example():
    """§6.4: zero input, causal, sq = sk = 2 -> [[1, 0], [0.5, 0.5]] (a wrong
    triangle, or a diagonal left out, changes it)."""
    want = np.loadtxt(GOLDEN, comments="#")
    got = O.scaled_masked_softmax_fwd(np.zeros((1, 2, 2), np.float32), 1.0, causal=True)[0]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n", [1, 5, 37])
def test_causal_zero_closed_form(n):
    """Row q of the causal softmax of zeros is 1/(q+1) on k <= q, 0 after."""
    got = O.scaled_masked_softmax_fwd(np.zeros((2, n, n), np.float32), 0.3, causal=True)
    q = np.arange(n)[:, None]
    k = np.arange(n)[None, :]
    want = np.where(k <= q, 1.0 / (q + 1), 0.0)
    assert np.allclose(got, want[None], rtol=1e-15, atol=0)


@pytest.mark.parametrize("scale", [1.0, 0.125, 1 / np.sqrt(128), 3.7])
@pytest.mark.parametrize("shape", [(3, 5, 7), (2, 3, 4, 33), (1, 1, 1, 1)])
def test_unmasked_equals_scipy(scale, shape):
    """No mask: scipy's softmax of scale * x (catches a missing or inverted
    scale and a wrong reduction axis)."""
    x = _x(shape, 1, 2.0)
    got = O.scaled_masked_softmax_fwd(x, scale)
    want = sp_softmax(x.astype(np.float64) * np.float64(np.float32(scale)), axis=-1)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-300)


def test_bf16_input_equals_scipy_of_widened_values():
    x = W.normal((2, 3, 5, 40), torch.bfloat16, 3)
    got = O.scaled_masked_softmax_fwd(W.to_oracle(x), 0.5)
    want = sp_softmax(x.double().numpy() * 0.5, axis=-1)
    assert np.allclose(got, want, rtol=1e-13, atol=0)


@pytest.mark.parametrize("mshape", [(1, 1, 6, 9), (2, 1, 1, 9), (2, 3, 6, 9), (1, 3, 1, 9), (2, 1, 6, 9)])
def test_additive_mask_broadcast_equals_numpy(mshape):
    """scale * x + mask with numpy's broadcasting of a [mb, mnp, msq, sk]
    mask, then scipy's softmax (catches a mask added before the scale, and a
    mask row taken from the wrong batch, head or query)."""
    x = _x((2, 3, 6, 9), 4)
    mask = _x(mshape, 5, 3.0)
    got = O.scaled_masked_softmax_fwd(x, 0.7, mask=mask)
    z = x.astype(np.float64) * np.float64(np.float32(0.7)) + np.broadcast_to(mask, x.shape).astype(np.float64)
    assert np.allclose(got, sp_softmax(z, axis=-1), rtol=1e-13, atol=0)


def test_minus_inf_mask_excludes_positions():
    """-inf entries: exactly 0 there, and the softmax of the remaining
    positions elsewhere."""
    x = _x((1, 2, 4, 11), 6)
    keep = np.random.default_rng(7).random((1, 1, 4, 11)) < 0.6
    keep[..., 0] = True
    mask = np.where(keep, 0.0, -np.inf).astype(np.float32)
    got = O.scaled_masked_softmax_fwd(x, 1.3, mask=mask)
    kb = np.broadcast_to(keep, x.shape)
    assert np.all(got[~kb] == 0.0)
    for h in range(2):
        for q in range(4):
            sel = keep[0, 0, q]
            want = sp_softmax(x[0, h, q, sel].astype(np.float64) * np.float64(np.float32(1.3)))
            assert np.allclose(got[0, h, q, sel], want, rtol=1e-13, atol=0)


def test_causal_equals_upper_triangle_minus_inf_mask_and_prefix_softmax():
    """Causal: the same as an additive mask with -inf strictly above the
    diagonal, and row q equals the softmax of the prefix k <= q."""
    n = 13
    x = _x((4, n, n), 8)
    got = O.scaled_masked_softmax_fwd(x, 0.9, causal=True)
    tri = np.triu(np.full((n, n), -np.inf, np.float32), k=1)[None, None]
    viamask = O.scaled_masked_softmax_fwd(x[None], 0.9, mask=tri)[0]
    assert np.array_equal(got, viamask)
    for q in range(n):
        want = sp_softmax(x[:, q, :q + 1].astype(np.float64) * np.float64(np.float32(0.9)), axis=-1)
        assert np.allclose(got[:, q, :q + 1], want, rtol=1e-13, atol=0)
        assert np.all(got[:, q, q + 1:] == 0.0)


def test_fully_masked_row_is_zero():
    """The reading for a row with no position left: zeros (not NaN)."""
    x = _x((1, 1, 3, 5), 9)
    mask = np.zeros((1, 1, 3, 5), np.float32)
    mask[0, 0, 1, :] = -np.inf
    got = O.scaled_masked_softmax_fwd(x, 1.0, mask=mask)
    assert np.all(got[0, 0, 1] == 0.0)
    assert np.allclose(got[0, 0, [0, 2]].sum(-1), 1.0, rtol=1e-15)


def test_nan_and_inf_rows_follow_torch():
    """A NaN score, or a +inf one, makes the row NaN, as torch's float64
    softmax does."""
    x = _x((3, 6), 10)
    x[0, 2] = np.nan
    x[1, 4] = np.inf
    got = O.scaled_masked_softmax_fwd(x, 1.0)
    want = torch.softmax(torch.from_numpy(x.astype(np.float64)), dim=-1).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.allclose(got[2], want[2], rtol=1e-13)


def test_rows_sum_to_one_and_shift_invariance():
    x = _dyadic((2, 2, 8, 300), 11) * np.float32(4.0)
    y = O.scaled_masked_softmax_fwd(x, 0.25)
    assert np.allclose(y.sum(-1), 1.0, rtol=1e-13)
    y2 = O.scaled_masked_softmax_fwd(x + np.float32(8.0), 0.25)  # exact shift of the dyadic range
    assert np.allclose(y, y2, rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_is_vjp_of_forward(causal):
    """dx equals central differences of sum(dy * forward(x)) (catches a
    missing scale, a wrong sign, the row sum taken without y, and a causal
    gradient leaking into excluded positions)."""
    n, scale = 5, 0.75
    x = _dyadic((2, n, n), 12)
    dy = _x((2, n, n), 13)
    y = O.scaled_masked_softmax_fwd(x, scale, causal=causal).astype(np.float32)
    dx = O.scaled_softmax_bwd(dy, y, scale, causal=causal)
    h = np.float32(2.0 ** -12)
    dyd = dy.astype(np.float64)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = ((dyd * O.scaled_masked_softmax_fwd(xp, scale, causal=causal)).sum() -
              (dyd * O.scaled_masked_softmax_fwd(xm, scale, causal=causal)).sum()) / (2 * np.float64(h))
        assert abs(dx[idx] - fd) <= 2e-6 * max(1.0, abs(fd)), (idx, dx[idx], fd)


def test_backward_identities():
    """Rows of dx sum to 0 (the softmax Jacobian annihilates constants), dx is
    linear in scale and in dy, and positions with y = 0 get 0."""
    x = _x((4, 64), 14)
    y = O.scaled_masked_softmax_fwd(x, 1.0).astype(np.float32)
    y[0, :10] = 0.0
    dy = _x((4, 64), 15)
    dx, sc = O.scaled_softmax_bwd(dy, y, 0.5, with_scale=True)
    s = (dy.astype(np.float64) * y).sum(-1, keepdims=True)
    # the row sum of dx is scale * s * (1 - sum y): zero up to the rounding of y
    assert np.allclose(dx.sum(-1), 0.5 * s[:, 0] * (1.0 - y.astype(np.float64).sum(-1)), atol=1e-13)
    assert np.array_equal(dx[0, :10], np.zeros(10))
    dx2 = O.scaled_softmax_bwd(dy, y, 1.0)
    assert np.allclose(dx2, 2.0 * dx, rtol=1e-15, atol=0)
    dx3 = O.scaled_softmax_bwd((dy * np.float32(2.0)).astype(np.float32), y, 0.5)
    assert np.allclose(dx3, 2.0 * dx, rtol=1e-15, atol=0)
    assert np.all(np.abs(dx) <= sc * (1 + 1e-15))


def test_backward_causal_zero_and_bf16():
    """Causal: excluded positions are exactly 0 even where dy is not finite;
    bf16 inputs are read as their widened values."""
    n = 6
    x = W.normal((2, n, n), torch.bfloat16, 16)
    y = torch.from_numpy(O.scaled_masked_softmax_fwd(W.to_oracle(x), 1.0, causal=True)).to(torch.bfloat16)
    dy = W.normal((2, n, n), torch.bfloat16, 17)
    dy[:, 0, n - 1] = float("inf")
    dy[:, 2, 3] = float("inf")  # just above the diagonal
    dx = O.scaled_softmax_bwd(W.to_oracle(dy), W.to_oracle(y), 2.0, causal=True)
    tri = np.triu(np.ones((n, n), bool), k=1)
    assert np.all(dx[:, tri] == 0.0)
    yd, gd = y.double().numpy(), dy.double().numpy()
    gd[:, tri] = 0.0  # the excluded positions take no part
    s = (gd * yd).sum(-1, keepdims=True)
    want = np.where(tri, 0.0, 2.0 * yd * (gd - s))
    assert np.allclose(dx, want, rtol=1e-15, atol=0)
