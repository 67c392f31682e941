"""Parity of the scale-mask-softmax kernels (through the C ABI) with the CPU
oracle: every team width of the register kernels and the long-row kernel,
ragged row lengths, padding, broadcast and causal masks, in-place and
misaligned buffers, rows with nothing left, extreme scores and the
determinism of the row reductions.  Tolerances: tests/parity.py (bf16: 1 ulp;
fp32: 1e-6 or 2 ulps; the backward adds the condition term of dy - sum)."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bits, check

pytestmark = pytest.mark.gpu

DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16]
BF16 = torch.bfloat16

# (b, np, sq, sk): sk spans team widths 1 .. 256 threads (4 chunks of 8 per
# thread), ragged lengths, the largest register row (8192) and the long-row
# kernel (8200, 20000).
SHAPES = [(1, 1, 1, 1), (2, 1, 3, 7), (1, 2, 5, 16), (2, 3, 4, 31), (1, 2, 9, 100), (2, 2, 8, 128),
          (1, 3, 7, 257), (2, 1, 6, 1000), (1, 2, 5, 1024), (1, 1, 9, 4096), (1, 1, 4, 4099),
          (1, 1, 3, 8192), (1, 1, 3, 8200), (1, 1, 3, 16384), (1, 1, 2, 16392), (1, 1, 2, 20000),
          (3, 4, 37, 64)]


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


def _oracle_y(x, scale, mask=None, causal=False):
    """The forward's output as the backward's input: the oracle's softmax,
    rounded to x's dtype on the host."""
    y = O.scaled_masked_softmax_fwd(W.to_oracle(x), scale, mask=W.to_oracle(mask), causal=causal)
    return torch.from_numpy(y).to(x.dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mask", [None, "pad", "full"])
def test_scaled_masked_softmax(dtype, shape, mask):
    b, np_, sq, sk = shape
    x, m, dy, scale = W.softmax_inputs(b, np_, sq, sk, dtype, seed=b * 1000 + sq * 31 + sk, mask=mask)
    ref = O.scaled_masked_softmax_fwd(W.to_oracle(x), scale, mask=W.to_oracle(m))
    y = mfx.mfx_scaled_masked_softmax_fwd(on(x), scale, on(m))
    yin = _oracle_y(x, scale, m)
    rdx, sc = O.scaled_softmax_bwd(W.to_oracle(dy), W.to_oracle(yin), scale, with_scale=True)
    dx = mfx.mfx_scaled_masked_softmax_bwd(on(dy), on(yin), scale)
    torch.cuda.synchronize()
    check(y, ref, f"softmax fwd {dtype} {shape} {mask}")
    check(dx, rdx, f"softmax bwd {dtype} {shape} {mask}", sc)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("ab,sq", [(1, 1), (2, 2), (3, 5), (2, 64), (1, 300), (2, 1030), (3, 512), (2, 1032),
                                   (1, 4096), (1, 8200)])
def test_causal_softmax(dtype, ab, sq):
    if sq == 8200 and dtype != BF16:
        pytest.skip("one long causal case is enough")
    x, _, dy, scale = W.softmax_inputs(1, ab, sq, sq, dtype, seed=ab * 7 + sq)
    x, dy = x[0], dy[0]
    ref = O.scaled_masked_softmax_fwd(W.to_oracle(x), scale, causal=True)
    y = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(on(x), scale)
    yin = _oracle_y(x, scale, causal=True)
    rdx, sc = O.scaled_softmax_bwd(W.to_oracle(dy), W.to_oracle(yin), scale, causal=True, with_scale=True)
    dx = mfx.mfx_scaled_upper_triang_masked_softmax_bwd(on(dy), on(yin), scale)
    torch.cuda.synchronize()
    check(y, ref, f"causal fwd {dtype} {ab}x{sq}")
    check(dx, rdx, f"causal bwd {dtype} {ab}x{sq}", sc)
    tri = torch.triu(torch.ones(sq, sq, dtype=torch.bool), diagonal=1)
    assert np.all(bits(y.cpu()[:, tri]) == 0) and np.all(bits(dx.cpu()[:, tri]) == 0)


def test_page_causal_zero_example():
    """The page's fallback test: zero input, causal, sq = sk = 2."""
    for dtype in DTYPES:
        y = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(torch.zeros(1, 2, 2, dtype=dtype, device=DEV), 1.0)
        assert torch.equal(y.cpu().float(), torch.tensor([[[1.0, 0.0], [0.5, 0.5]]]))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("sk", [24, 1024, 20000])
def test_misaligned_and_in_place_match_aligned(dtype, sk):
    x, m, dy, scale = W.softmax_inputs(2, 2, 3, sk, dtype, seed=sk, mask="pad")
    xd, md, dyd = on(x), on(m), on(dy)
    y = mfx.mfx_scaled_masked_softmax_fwd(xd, scale, md)
    ym = mfx.mfx_scaled_masked_softmax_fwd(misaligned(x), scale, misaligned(m), y=misaligned(torch.zeros_like(x)))
    xi = xd.clone()
    yi = mfx.mfx_scaled_masked_softmax_fwd(xi, scale, md, y=xi)
    yin = on(_oracle_y(x, scale, m))
    dx = mfx.mfx_scaled_masked_softmax_bwd(dyd, yin, scale)
    dxm = mfx.mfx_scaled_masked_softmax_bwd(misaligned(dy), misaligned(yin.cpu()), scale,
                                            dx=misaligned(torch.zeros_like(x)))
    g2 = dyd.clone()
    dxi = mfx.mfx_scaled_masked_softmax_bwd(g2, yin, scale, dx=g2)
    y2 = yin.clone()
    dxy = mfx.mfx_scaled_masked_softmax_bwd(dyd, y2, scale, dx=y2)
    torch.cuda.synchronize()
    for other in (ym, yi):
        assert np.array_equal(bits(y), bits(other))
    for other in (dxm, dxi, dxy):
        assert np.array_equal(bits(dx), bits(other))


def test_causal_misaligned_and_in_place_match_aligned():
    x, _, dy, scale = W.softmax_inputs(1, 3, 40, 40, BF16, seed=9)
    x, dy = x[0], dy[0]
    y = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(on(x), scale)
    ym = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(misaligned(x), scale, y=misaligned(torch.zeros_like(x)))
    xi = on(x)
    yi = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(xi, scale, y=xi)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), bits(ym)) and np.array_equal(bits(y), bits(yi))


@pytest.mark.parametrize("dtype", DTYPES)
def test_causal_pipeline_in_place_matches(dtype):
    """Row lengths the pipelined causal kernels take (rows paired within each
    head): in-place forward and backward give the out-of-place bits."""
    x, _, dy, scale = W.softmax_inputs(1, 3, 520, 520, dtype, seed=21)
    x, dy = on(x[0]), on(dy[0])
    y = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(x, scale)
    yi = x.clone()
    mfx.mfx_scaled_upper_triang_masked_softmax_fwd(yi, scale, y=yi)
    dx = mfx.mfx_scaled_upper_triang_masked_softmax_bwd(dy, y, scale)
    dxi = dy.clone()
    mfx.mfx_scaled_upper_triang_masked_softmax_bwd(dxi, y, scale, dx=dxi)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), bits(yi)) and np.array_equal(bits(dx), bits(dxi))


@pytest.mark.parametrize("dtype", DTYPES)
def test_broadcast_masks_equal_expanded(dtype):
    """Each broadcast form gives the same bits as the mask expanded to x's
    shape."""
    x, _, _, scale = W.softmax_inputs(2, 3, 5, 40, dtype, seed=11)
    full = W.normal((2, 3, 5, 40), dtype, 12)
    xd = on(x)
    for mshape in [(1, 1, 1, 40), (2, 1, 1, 40), (1, 3, 1, 40), (1, 1, 5, 40), (2, 3, 1, 40), (2, 1, 5, 40)]:
        sl = tuple(slice(0, n) for n in mshape)
        m = full[sl].contiguous()
        y = mfx.mfx_scaled_masked_softmax_fwd(xd, scale, on(m))
        ye = mfx.mfx_scaled_masked_softmax_fwd(xd, scale, on(m.expand(2, 3, 5, 40).contiguous()))
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), bits(ye)), mshape


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("sk", [40, 20000])
def test_rows_with_nothing_left_are_zero(dtype, sk):
    x, _, dy, scale = W.softmax_inputs(1, 2, 4, sk, dtype, seed=13)
    m = torch.zeros(1, 1, 4, sk)
    m[0, 0, 1, :] = float("-inf")
    x[0, 1, 2, :] = float("-inf")           # scores themselves -inf
    x[0, 0, 3, :] = float("nan")            # NaN scores with a -inf mask: still nothing left
    m[0, 0, 3, :] = float("-inf")
    m = m.to(dtype)
    ref = O.scaled_masked_softmax_fwd(W.to_oracle(x), scale, mask=W.to_oracle(m))
    y = mfx.mfx_scaled_masked_softmax_fwd(on(x), scale, on(m))
    torch.cuda.synchronize()
    check(y, ref, f"empty rows {dtype} {sk}")
    yc = y.cpu()
    assert np.all(bits(yc[0, :, 1]) == 0) and np.all(bits(yc[0, 1, 2]) == 0) and np.all(bits(yc[0, :, 3]) == 0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_extreme_scores(dtype):
    """Large finite scores (the exponent keeps its accuracy), spreads that
    reach the smallest subnormal outputs, NaN and +inf scores (NaN rows),
    and an infinite upstream gradient."""
    sk = 64
    rows = []
    rows.append(torch.linspace(-1e30, 1e30, sk))                 # one winner, huge scores
    rows.append(torch.linspace(1000.0, 1001.0, sk))              # large offset, small spread
    rows.append(torch.linspace(-200.0, 0.0, sk))                 # outputs down to e^-200
    rows.append(torch.linspace(-95.0, -80.0, sk))
    r = torch.randn(sk, generator=W.gen(3))
    r[5] = float("nan")
    rows.append(r)
    r = torch.randn(sk, generator=W.gen(4))
    r[9] = float("inf")
    rows.append(r)
    rows.append(torch.full((sk,), 3e38))                         # equal huge scores: uniform
    x = torch.stack(rows)[None, None].to(dtype)
    ref = O.scaled_masked_softmax_fwd(W.to_oracle(x), 1.0)
    y = mfx.mfx_scaled_masked_softmax_fwd(on(x), 1.0)
    dy = torch.randn(x.shape, generator=W.gen(5)).to(dtype)
    yin = _oracle_y(x, 1.0)[..., :3, :].contiguous()
    dyb = dy[..., :3, :].contiguous()
    dyb[0, 0, 2, 7] = float("inf")
    rdx, sc = O.scaled_softmax_bwd(W.to_oracle(dyb), W.to_oracle(yin), 1.0, with_scale=True)
    dx = mfx.mfx_scaled_masked_softmax_bwd(on(dyb), on(yin), 1.0)
    torch.cuda.synchronize()
    check(y, ref, f"softmax extremes {dtype}")
    check(dx, rdx, f"softmax bwd extremes {dtype}", sc)


def test_reductions_are_deterministic():
    x, m, dy, scale = W.softmax_inputs(2, 4, 16, 4099, BF16, seed=21, mask="pad")
    xd, md, dyd = on(x), on(m), on(dy)
    ys = [mfx.mfx_scaled_masked_softmax_fwd(xd, scale, md).clone() for _ in range(3)]
    dxs = [mfx.mfx_scaled_masked_softmax_bwd(dyd, ys[0], scale).clone() for _ in range(3)]
    torch.cuda.synchronize()
    for a in ys[1:]:
        assert np.array_equal(bits(ys[0]), bits(a))
    for a in dxs[1:]:
        assert np.array_equal(bits(dxs[0]), bits(a))


def test_argument_errors():
    L = mfx.lib()
    x = torch.zeros(2, 3, 4, 8, dtype=BF16, device=DEV)
    m = torch.zeros(2, 2, 4, 8, dtype=BF16, device=DEV)     # 2 heads where x has 3
    y = torch.empty_like(x)
    assert L.mfx_scaled_masked_softmax_fwd(1, 2, 3, 4, 8, x.data_ptr(), m.data_ptr(), 2, 2, 4, 1.0,
                                           y.data_ptr(), None) == 2
    assert L.mfx_scaled_masked_softmax_fwd(1, 2, 3, 4, 8, x.data_ptr(), None, 2, 2, 4, 1.0,
                                           y.data_ptr(), None) == 0  # no mask: its sizes are ignored
    assert L.mfx_scaled_masked_softmax_fwd(1, 2, 3, 4, 8, x.data_ptr(), None, 1, 1, 1, 1.0,
                                           x.data_ptr() + 2, None) == 5
    assert L.mfx_scaled_masked_softmax_fwd(7, 2, 3, 4, 8, None, None, 1, 1, 1, 1.0, None, None) == 3
    assert L.mfx_scaled_masked_softmax_fwd(1, 0, 3, 4, 8, None, None, 1, 1, 1, 1.0, None, None) == 0
    assert L.mfx_scaled_upper_triang_masked_softmax_bwd(1, -1, 4, None, None, 1.0, None, None) == 2
    assert L.mfx_scaled_masked_softmax_bwd(1, 4, 8, x.data_ptr(), None, 1.0, y.data_ptr(), None) == 1
    with pytest.raises(ValueError):
        mfx.mfx_scaled_upper_triang_masked_softmax_fwd(torch.zeros(2, 3, 4, device=DEV), 1.0)
    torch.cuda.synchronize()
