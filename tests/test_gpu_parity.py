"""Parity of the CUDA kernels (called through the C ABI) with the CPU oracle
on small and ragged shapes, misaligned buffers, in-place calls and extreme
values.  Tolerances: tests/parity.py."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bits, check, check_bf16, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16]
BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def on(t):
    return None if t is None else t.to(DEV)


def misaligned(t):
    """The same values at an address one element past a 16-byte boundary."""
    if t is None:
        return None
    buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0 and v.is_contiguous()
    return v


def sync():
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# bias-GeLU
# ---------------------------------------------------------------------------
GELU_SHAPES = [(1, 1), (1, 7), (2, 9), (3, 4099), (17, 24), (64, 1024), (33, 4104), (5, 16384)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", GELU_SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_bias_gelu(dtype, shape, with_bias):
    rows, cols = shape
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=rows * 131 + cols, with_bias=with_bias)
    ref_f = O.bias_gelu_fwd(W.to_oracle(y), W.to_oracle(b))
    ref_b, scale = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b), with_scale=True)
    out = mfx.mfx_bias_gelu_fwd(on(b), on(y))
    dy = mfx.mfx_bias_gelu_bwd(on(g), on(b), on(y))
    sync()
    check(out, ref_f, f"gelu fwd {dtype} {shape}")
    check(dy, ref_b, f"gelu bwd {dtype} {shape}", scale)


@pytest.mark.parametrize("dtype", DTYPES)
def test_bias_gelu_misaligned_and_in_place_match_aligned(dtype):
    """The generic path (misaligned buffers) and in-place calls give the same
    bits as the aligned fast path."""
    y, b, g = W.gelu_inputs(24, 4096, dtype, seed=5)
    yd, bd, gd = on(y), on(b), on(g)
    out = mfx.mfx_bias_gelu_fwd(bd, yd)
    dy = mfx.mfx_bias_gelu_bwd(gd, bd, yd)
    out_m = mfx.mfx_bias_gelu_fwd(misaligned(b), misaligned(y), out=misaligned(torch.zeros_like(y)))
    dy_m = mfx.mfx_bias_gelu_bwd(misaligned(g), misaligned(b), misaligned(y),
                                 dy=misaligned(torch.zeros_like(y)))
    inplace = yd.clone()
    mfx.mfx_bias_gelu_fwd(bd, inplace, out=inplace)
    g_inplace = gd.clone()
    mfx.mfx_bias_gelu_bwd(g_inplace, bd, yd, dy=g_inplace)
    sync()
    for a, c in [(out, out_m), (out, inplace), (dy, dy_m), (dy, g_inplace)]:
        assert np.array_equal(bits(a), bits(c))
    check(out, O.bias_gelu_fwd(W.to_oracle(y), W.to_oracle(b)))


@pytest.mark.parametrize("dtype", DTYPES)
def test_bias_gelu_extreme_values(dtype):
    """A dense sweep over [-12, 12] (far tails where 1 + tanh u underflows),
    huge magnitudes whose square overflows fp32, zeros and infinities."""
    sweep = torch.linspace(-12, 12, 24 * 1024)
    special = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e20, -1e20, 3e38, -3e38,
                            float("inf"), float("-inf"), 9.5, -9.5, 10.5, -10.5, 30.0, -30.0])
    y = torch.cat([sweep, special, torch.zeros(8 - special.numel() % 8)]).reshape(-1, 8).to(dtype)
    g = torch.ones_like(y)
    finite = torch.isfinite(y.float())
    ref_f = O.bias_gelu_fwd(W.to_oracle(y))
    ref_b, scale = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), with_scale=True)
    out = mfx.mfx_bias_gelu_fwd(None, on(y))
    dy = mfx.mfx_bias_gelu_bwd(on(g), None, on(y))
    sync()
    check(out, ref_f, "gelu fwd extremes")
    fin = finite.numpy()
    check(dy.cpu()[finite], ref_b[fin], "gelu bwd extremes", scale[fin])
    assert torch.isnan(dy.cpu()[~finite].float()).all()


# ---------------------------------------------------------------------------
# GEGLU / SwiGLU
# ---------------------------------------------------------------------------
GLU_SHAPES = [(1, 1), (2, 3), (3, 8), (5, 13), (7, 1024), (3, 4099), (2, 14336), (9, 40), (13, 2400),
              (6, 264)]


def _glu_ref(kind, x, b, g, w):
    """(fwd, dx, dweight, dweight_abs, dx condition scale) from the oracle."""
    xo, bo, go, wo = W.to_oracle(x), W.to_oracle(b), W.to_oracle(g), W.to_oracle(w)
    if kind == "geglu":
        dx, sc = O.bias_geglu_bwd(go, xo, bo, with_scale=True)
        return O.bias_geglu_fwd(xo, bo), dx, None, None, sc
    f = O.bias_swiglu_fwd(xo, bo, wo)
    dx, dw, dwa, sc = O.bias_swiglu_bwd(go, xo, bo, wo, with_scale=True)
    return f, dx, dw, dwa, sc


def _glu_gpu(kind, x, b, g, w, out=None, dx=None):
    if kind == "geglu":
        return mfx.mfx_bias_geglu_fwd(x, b, out=out), mfx.mfx_bias_geglu_bwd(g, x, b, dx=dx), None
    f = mfx.mfx_bias_swiglu_fwd(x, b, w, out=out)
    d, dw = mfx.mfx_bias_swiglu_bwd(g, x, b, w, dx=dx)
    return f, d, dw


def check_dweight(dw, ref, ref_abs, what):
    """Weight gradient (an fp32 row sum): |err| <= 1e-5 * sum_c |term|."""
    err = np.abs(to_f64(dw) - ref)
    assert np.all(err <= 1e-5 * ref_abs + 1e-30), f"{what}: max rel-to-abs-sum {np.max(err / ref_abs):.3e}"


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", GLU_SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_glu(kind, dtype, shape, with_bias):
    rows, F = shape
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=rows * 17 + F, with_bias=with_bias,
                              with_weight=kind == "swiglu_w")
    ref_f, ref_dx, ref_dw, ref_dwa, sc = _glu_ref(kind, x, b, g, w)
    f, dx, dw = _glu_gpu(kind, on(x), on(b), on(g), on(w))
    sync()
    check(f, ref_f, f"{kind} fwd {dtype} {shape}")
    check(dx, ref_dx, f"{kind} bwd {dtype} {shape}", sc)
    if kind == "swiglu_w":
        check_dweight(dw, ref_dw, ref_dwa, f"{kind} dweight {dtype} {shape}")


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_glu_misaligned_and_in_place_match_aligned(kind, dtype):
    rows, F = 6, 1024
    x, b, g, w = W.glu_inputs(rows, F, dtype, seed=3, with_weight=kind == "swiglu_w")
    xd, bd, gd, wd = on(x), on(b), on(g), on(w)
    f, dx, dw = _glu_gpu(kind, xd, bd, gd, wd)
    fm, dxm, dwm = _glu_gpu(kind, misaligned(x), misaligned(b), misaligned(g), wd,
                            out=misaligned(torch.zeros(rows, F, dtype=dtype)),
                            dx=misaligned(torch.zeros_like(x)))
    xi = xd.clone()
    _, dxi, dwi = _glu_gpu(kind, xi, bd, gd, wd, dx=xi)
    sync()
    assert np.array_equal(bits(f), bits(fm))
    assert np.array_equal(bits(dx), bits(dxm))
    assert np.array_equal(bits(dx), bits(dxi))
    if dw is not None:
        assert np.array_equal(bits(dw), bits(dwm)) and np.array_equal(bits(dw), bits(dwi))


@pytest.mark.parametrize("dtype", DTYPES)
def test_weighted_swiglu_identity(dtype):
    """weighted(x, w) matches swiglu(x) * w, the page's weighted-SwiGLU test
    (fusions page §9).  Both sides are outputs held to their own gates, so the
    bound is the weighted output's (1 ulp at the product's binade; 2 in fp32,
    for its internal roundings) plus the unweighted output's scaled by w: 1
    bf16 ulp (its gate: the bf16 forward's reciprocal may spend up to 0.45 ulp
    before the final rounding), half an fp32 ulp (the precise tier rounds
    once)."""
    from parity import bf16_ulp, f32_ulp
    x, b, g, w = W.glu_inputs(64, 1024, dtype, seed=8, with_weight=True)
    xd, bd, wd = on(x), on(b), on(w)
    weighted = mfx.mfx_bias_swiglu_fwd(xd, bd, wd)
    plain = mfx.mfx_bias_swiglu_fwd(xd, bd)
    sync()
    wv = to_f64(wd)[:, None]
    pv = to_f64(plain)
    prod = pv * wv
    ulp = bf16_ulp if dtype == BF16 else f32_ulp
    k, kp = (1.0, 1.0) if dtype == BF16 else (2.0, 0.5)
    tol = k * ulp(prod) + kp * ulp(pv) * wv
    assert np.all(np.abs(to_f64(weighted) - prod) <= tol)


def test_weighted_swiglu_dweight_is_deterministic():
    x, b, g, w = W.glu_inputs(300, 4104, BF16, seed=4, with_weight=True)
    xd, bd, gd, wd = on(x), on(b), on(g), on(w)
    outs = [mfx.mfx_bias_swiglu_bwd(gd, xd, bd, wd)[1].clone() for _ in range(3)]
    sync()
    for o in outs[1:]:
        assert np.array_equal(bits(outs[0]), bits(o))


@pytest.mark.parametrize("dtype", DTYPES)
def test_glu_extreme_values(dtype):
    a = torch.cat([torch.linspace(-40, 40, 4000), torch.tensor([1e20, -1e20, 0.0, -0.0, 3e38, -3e38, 88.0, -88.0])])
    F = a.numel()
    x = torch.stack([torch.cat([a, torch.full((F,), 1.5)]), torch.cat([a, -a])]).to(dtype)
    g = torch.ones(2, F).to(dtype)
    for kind in ("geglu", "swiglu"):
        ref_f, ref_dx, _, _, sc = _glu_ref(kind, x, None, g, None)
        f, dx, _ = _glu_gpu(kind, on(x), None, on(g), None)
        sync()
        check(f, ref_f, f"{kind} fwd extremes {dtype}")
        check(dx, ref_dx, f"{kind} bwd extremes {dtype}", sc)


# ---------------------------------------------------------------------------
# bias-dropout-add
# ---------------------------------------------------------------------------
COMBOS = [(BF16, F32), (BF16, BF16), (F32, F32), (F32, BF16)]
BDA_SHAPES = [(1, 1), (1, 7), (2, 9), (3, 4099), (5, 24), (16, 4096)]


@pytest.mark.parametrize("xdt,rdt", COMBOS)
@pytest.mark.parametrize("shape", BDA_SHAPES)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("elem_base", [0, 5, 8 * 1000 + 3])
def test_dropout_train_bit_exact(xdt, rdt, shape, p, elem_base):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + cols)
    seed, offset = 1234 + (5 << 40), 7 + (3 << 33)
    ref_out, ref_keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=p,
                                                 seed=seed, offset=offset, elem_base=elem_base)
    out, keep = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), p, seed, offset, elem_base)
    sync()
    assert np.array_equal(keep.cpu().numpy(), ref_keep)
    assert np.array_equal(bits(out), ref_out.view(bits(out).dtype))


@pytest.mark.parametrize("xdt,rdt", COMBOS)
@pytest.mark.parametrize("shape", BDA_SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_dropout_inference_in_place_bit_exact(xdt, rdt, shape, with_bias):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows * 3 + cols, with_bias=with_bias)
    ref = W.to_oracle(x)
    O.bias_dropout_add_inference(ref, W.to_oracle(r), W.to_oracle(b))
    xd = on(x)
    ptr = xd.data_ptr()
    ret = mfx.mfx_bias_dropout_add_inference(xd, on(b), on(r), 0.1, 1234, 0)
    sync()
    assert ret.data_ptr() == ptr == xd.data_ptr()   # in place (the page's data_ptr check)
    assert np.array_equal(bits(xd), ref.view(bits(xd).dtype))


@pytest.mark.parametrize("xdt,rdt", COMBOS)
def test_dropout_paths_agree(xdt, rdt):
    """Aligned fast path, misaligned generic path, out == x, and two half
    calls with their own elem_base all give the same bits."""
    rows, cols = 32, 4096
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=11)
    xd, bd, rd = on(x), on(b), on(r)
    out, keep = mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.3, 99, 5, 0)
    out_m, keep_m = mfx.mfx_bias_dropout_add_train(
        misaligned(x), misaligned(b), misaligned(r), 0.3, 99, 5, 0,
        out=misaligned(torch.zeros_like(x)),
        keep_mask=misaligned(torch.zeros(rows, cols, dtype=torch.uint8)))
    xi = xd.clone()
    out_i, keep_i = mfx.mfx_bias_dropout_add_train(xi, bd, rd, 0.3, 99, 5, 0, out=xi)
    h = rows // 2
    top = mfx.mfx_bias_dropout_add_train(xd[:h], bd, rd[:h], 0.3, 99, 5, 0)
    bot = mfx.mfx_bias_dropout_add_train(xd[h:], bd, rd[h:], 0.3, 99, 5, h * cols)
    sync()
    for o, k in [(out_m, keep_m), (out_i, keep_i)]:
        assert np.array_equal(bits(out), bits(o)) and np.array_equal(bits(keep), bits(k))
    assert np.array_equal(bits(out), np.concatenate([bits(top[0]), bits(bot[0])]))
    assert np.array_equal(bits(keep), np.concatenate([bits(top[1]), bits(bot[1])]))


def test_dropout_p0_keeps_everything():
    x, b, r = W.dropout_inputs(64, 4096, BF16, F32, seed=2)
    out, keep = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), 0.0, 1, 0, 0)
    sync()
    assert bool(keep.all())


def test_dropout_mask_depends_on_seed_and_offset():
    x, b, r = W.dropout_inputs(64, 4096, BF16, F32, seed=2)
    xd, bd, rd = on(x), on(b), on(r)
    k0 = mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.5, 1234, 0)[1]
    k1 = mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.5, 1235, 0)[1]
    k2 = mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.5, 1234, 1)[1]
    sync()
    n = k0.numel()
    for k in (k1, k2):
        frac = (k0 != k).float().mean().item()
        assert abs(frac - 0.5) < 4 * (0.25 / n) ** 0.5


def test_empty_tensors_are_no_ops():
    e = torch.empty(0, 16, device=DEV, dtype=BF16)
    assert mfx.mfx_bias_gelu_fwd(None, e).numel() == 0
    assert mfx.mfx_bias_swiglu_fwd(e, None).shape == (0, 8)
    out, keep = mfx.mfx_bias_dropout_add_train(e, None, e.float(), 0.1, 1, 0)
    assert out.numel() == 0 and keep.numel() == 0
    sync()


def test_no_bounded_wait_ran_out():
    """The pipelined kernels' barrier waits never time out in these runs (the
    device error word is 0 and reading it clears it)."""
    x, b, r = W.dropout_inputs(64, 4096, BF16, F32, seed=2)
    mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), 0.1, 1, 0)
    mfx.mfx_bias_dropout_add_inference(on(x), on(b), on(r))
    xg, bg, gg, wg = W.glu_inputs(64, 2400, BF16, seed=3, with_weight=True)
    mfx.mfx_bias_swiglu_fwd(on(xg), on(bg), on(wg))
    mfx.mfx_bias_geglu_bwd(on(gg), on(xg), on(bg))
    y, by, gy = W.gelu_inputs(64, 4096, BF16, seed=4)
    mfx.mfx_bias_gelu_fwd(on(by), on(y))
    mfx.mfx_bias_gelu_bwd(on(gy), on(by), on(y))
    assert mfx.mfx_device_error() == 0
    assert mfx.lib().mfx_device_error(None) == 0


# ---------------------------------------------------------------------------
# bias-dropout-add backward (NEXT row f1)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("xdt,rdt", COMBOS)
@pytest.mark.parametrize("shape", BDA_SHAPES)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("elem_base", [0, 5])
@pytest.mark.parametrize("regen", [False, True])
def test_dropout_backward_bit_exact(xdt, rdt, shape, p, elem_base, regen):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + 3 * cols)
    g = W.normal((rows, cols), xdt, rows * 5 + cols)
    seed, offset = 99 + (1 << 35), 4
    _, keep = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), p, seed, offset, elem_base)
    dx, dres = mfx.mfx_bias_dropout_add_bwd(on(g), None if regen else keep, p, seed, offset, elem_base,
                                            residual_dtype=rdt)
    sync()
    rname = "bf16" if rdt == BF16 else "f32"
    ref_dx, ref_dres = O.bias_dropout_add_bwd(W.to_oracle(g), keep.cpu().numpy(), p=p, res_dtype=rname)
    assert np.array_equal(bits(dx), ref_dx.view(bits(dx).dtype))
    assert np.array_equal(bits(dres), ref_dres.view(bits(dres).dtype))
    # the forward's mask equals the oracle's regenerated one
    ref_dx2, _ = O.bias_dropout_add_bwd(W.to_oracle(g), None, p=p, seed=seed, offset=offset, elem_base=elem_base)
    assert np.array_equal(ref_dx, ref_dx2)


@pytest.mark.parametrize("xdt,rdt", COMBOS)
def test_dropout_backward_paths_agree(xdt, rdt):
    """Pipelined (aligned) and generic (misaligned) paths, in place, with and
    without the mask, give the same bits."""
    rows, cols = 24, 4096
    g = W.normal((rows, cols), xdt, 7)
    keep = (torch.rand(rows, cols) > 0.3).to(torch.uint8)
    gd, kd = on(g), on(keep)
    dx, dres = mfx.mfx_bias_dropout_add_bwd(gd, kd, 0.3, residual_dtype=rdt)
    dx_m, dres_m = mfx.mfx_bias_dropout_add_bwd(misaligned(g), misaligned(keep), 0.3,
                                                dx=misaligned(torch.zeros_like(g)),
                                                dresidual=misaligned(torch.zeros(rows, cols, dtype=rdt)))
    gi = gd.clone()
    dx_i, _ = mfx.mfx_bias_dropout_add_bwd(gi, kd, 0.3, dx=gi)
    sync()
    assert np.array_equal(bits(dx), bits(dx_m)) and np.array_equal(bits(dres), bits(dres_m))
    assert np.array_equal(bits(dx), bits(dx_i))
    assert mfx.mfx_device_error() == 0
