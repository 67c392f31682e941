"""Pins of the CPU oracle against things other than itself.

The oracle (oracle/mfx_oracle.c) restates the fused ops of the web page
"Megatron-LM operator fusion walkthrough" (www.wmrh.cn/news/51426).  Each test
below ties one oracle function to an independent source: the erf form of GeLU,
an arbitrary-precision evaluation of the printed formula, central finite
differences, scipy's logistic function, torch's bf16 rounding and fp32
arithmetic, and structural identities the page states.  The mistakes they are
chosen to catch are named in each docstring.
"""
import math
import os

import mpmath
import numpy as np
import pytest
import torch
from scipy.special import expit, ndtr

import oracle as O
from elementwise_epilogues_transformer_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gelu_constants.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, val, meaning, digits = line.split()
        out[name] = (float(val), meaning, int(digits))
    return out


# --------------------------------------------------------------------------
# bf16 conversions
# --------------------------------------------------------------------------
def test_bf16_decode_all_patterns_match_torch():
    """Widening every one of the 65536 bf16 patterns agrees with torch."""
    bits = np.arange(65536, dtype=np.uint16)
    ours = O.f32_from_bf16_bits(bits).view(np.uint32)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    ref = ref.view(np.uint32)
    nan = np.isnan(ours.view(np.float32))
    assert np.array_equal(nan, np.isnan(ref.view(np.float32)))
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_encode_is_round_nearest_even_like_torch():
    """Rounding fp32 -> bf16 agrees with torch on random values, exact ties,
    subnormals, overflow to inf and NaN (catches truncation or ties-away)."""
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(20000).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal
            np.array([3.3895e38, 3.4e38, -3.4e38, np.inf, -np.inf, 0.0, -0.0],
                     dtype=np.float32)]
    # exact ties: low 16 bits == 0x8000, with even and odd upper halves
    ties = (rng.integers(0, 2**15, 2000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32)
    vals.append(ties.view(np.float32))
    a = np.concatenate(vals)
    a = a[~np.isnan(a)]
    ours = O.bf16_bits_from_f32(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nan_bits = O.bf16_bits_from_f32(np.array([np.nan], dtype=np.float32))
    assert np.isnan(O.f32_from_bf16_bits(nan_bits)[0])


# --------------------------------------------------------------------------
# GeLU (tanh approximation, fusions page §4.2)
# --------------------------------------------------------------------------
def test_printed_constants_match_their_meaning():
    """Each constant the page prints equals the quantity it names, to the
    printed digits."""
    g = _golden()
    exact = {"1/sqrt(2*pi)": 1 / math.sqrt(2 * math.pi), "1/sqrt(2)": 1 / math.sqrt(2),
             "sqrt(2/pi)": math.sqrt(2 / math.pi),
             "3*0.79788456*0.044715": 3 * 0.79788456 * 0.044715}
    checked = 0
    for name, (val, meaning, digits) in g.items():
        if meaning in exact:
            ref = exact[meaning]
            half_unit = 0.5 * 10.0 ** (math.floor(math.log10(abs(ref))) - digits + 1)
            assert abs(val - ref) <= half_unit * (1 + 1e-9), name
            checked += 1
    assert checked == 4


def test_gelu_uses_printed_constants():
    """Recover the two constants of u = k0 x (1 + k1 x^2) from the oracle via
    gelu(h) + gelu(-h) = h tanh(u(h)) (tanh is odd), and compare with the
    printed values (catches a wrong or rounded constant)."""
    g = _golden()
    def q(h):
        s = (O.gelu_tanh(h) + O.gelu_tanh(-h)) / h
        return math.atanh(s) / h
    h1, h2 = 0.25, 0.5
    k0k1 = (q(h2) - q(h1)) / (h2 ** 2 - h1 ** 2)
    k0 = q(h1) - k0k1 * h1 ** 2
    k1 = k0k1 / k0
    assert abs(k0 - g["sqrt_2_over_pi"][0]) < 1e-10
    assert abs(k1 - g["cubic"][0]) < 1e-9


def test_gelu_close_to_exact_erf_gelu():
    """|gelu_tanh(x) - x Phi(x)| <= 5e-4 on [-10, 10], and the largest gap
    (near |x| = 2.7) is the tanh approximation's own, about 4.7e-4, not ~0
    (so the oracle is the tanh form, not the erf form the page calls exact)."""
    x = np.linspace(-10, 10, 20001)
    ours = np.array([O.lib().orc_gelu_tanh(float(v)) for v in x])
    d = np.abs(ours - x * ndtr(x))
    assert d.max() <= 5e-4
    assert 4.6e-4 <= d.max() <= 4.8e-4
    assert 2.6 <= abs(x[d.argmax()]) <= 2.8


def test_gelu_matches_arbitrary_precision_printed_formula():
    """The fp64 oracle, with its cancellation-free identities for 1 + tanh u
    and 1 - tanh^2 u, equals the printed formula evaluated with enough digits,
    to a few fp64 ulps (times |u|) in relative terms, including the far negative tail where
    the printed grouping cancels (catches a wrong identity or sign)."""
    for xv in list(np.linspace(-12, 12, 241)) + [-30.0, -20.0, 1e-6, -1e-6, 40.0]:
        # enough digits that 1 + tanh(u) ~ 2 e^(2u) survives the cancellation
        u_est = 0.8 * abs(xv) * (1 + 0.045 * xv * xv)
        mpmath.mp.dps = 40 + int(2 * u_est / math.log(10))
        k0, k1, kd = mpmath.mpf("0.79788456"), mpmath.mpf("0.044715"), mpmath.mpf("0.1070322243")
        x = mpmath.mpf(float(xv))
        u = k0 * x * (1 + k1 * x * x)
        t = mpmath.tanh(u)
        fwd = x * mpmath.mpf("0.5") * (1 + t)
        bwd = mpmath.mpf("0.5") * x * ((1 - t * t) * (k0 + kd * x * x)) + mpmath.mpf("0.5") * (1 + t)
        of, ob = O.gelu_tanh(float(xv)), O.gelu_tanh_grad(float(xv))
        for ours, ref in ((of, fwd), (ob, bwd)):
            ref = float(ref)
            if ref == 0.0:
                assert abs(ours) < 1e-300
            else:
                # e^(2u) turns the few-ulp rounding of u into ~|2u| ulps
                assert abs(ours - ref) <= (32 + 8 * u_est) * 2.0 ** -52 * abs(ref), (xv, ours, ref)


def test_gelu_special_values():
    assert O.gelu_tanh(0.0) == 0.0
    assert abs(O.gelu_tanh_grad(0.0) - 0.5) < 1e-15
    assert abs(O.gelu_tanh(20.0) - 20.0) < 1e-12
    assert -1e-30 < O.gelu_tanh(-20.0) <= 0.0


def test_gelu_odd_part_identity():
    """gelu(x) - gelu(-x) = x, because tanh is odd."""
    for x in np.linspace(-6, 6, 121):
        assert abs(O.gelu_tanh(x) - O.gelu_tanh(-x) - x) < 1e-13 * max(1, abs(x))


def test_gelu_backward_matches_central_differences():
    """The backward factor is the derivative of the forward (catches a wrong
    term or coefficient in the hand-derived backward)."""
    for x in np.linspace(-8, 8, 321):
        h = 1e-4 * max(1.0, abs(x))
        fd = (O.gelu_tanh(x + h) - O.gelu_tanh(x - h)) / (2 * h)
        assert abs(O.gelu_tanh_grad(x) - fd) <= 1e-7 * max(1.0, abs(x)) ** 3, x


# --------------------------------------------------------------------------
# logistic / SiLU
# --------------------------------------------------------------------------
def test_logistic_matches_scipy():
    z = np.concatenate([np.linspace(-60, 60, 2401), [-700.0, 700.0, 0.0]])
    ours = O.logistic(z)
    ref = expit(z)
    assert np.all(np.abs(ours - ref) <= 4 * np.finfo(np.float64).eps * np.abs(ref) + 1e-300)
    assert O.logistic(0.0) == 0.5


def test_silu_identities():
    for z in np.linspace(-10, 10, 201):
        assert abs(O.lib().orc_silu(z) - O.lib().orc_silu(-z) - z) < 1e-13 * max(1, abs(z))
    assert O.lib().orc_silu(0.0) == 0.0


# --------------------------------------------------------------------------
# tensor ops: bias add, GEGLU, SwiGLU
# --------------------------------------------------------------------------
def test_bias_add_is_one_fp32_addition():
    """With fp32 inputs the oracle's bias add is fl32(y + b): feeding the
    pre-rounded sum with no bias gives identical results."""
    y, b, _ = W.gelu_inputs(3, 37, torch.float32, seed=11)
    yn, bn = W.to_oracle(y), W.to_oracle(b)
    s = (yn + bn[None, :]).astype(np.float32)
    assert np.array_equal(O.bias_gelu_fwd(yn, bn), O.bias_gelu_fwd(s))
    g = W.to_oracle(torch.randn(3, 37))
    assert np.array_equal(O.bias_gelu_bwd(g, yn, bn), O.bias_gelu_bwd(g, s))


def test_bias_gelu_tensor_op_is_elementwise_gelu():
    y, b, g = W.gelu_inputs(4, 9, torch.bfloat16, seed=3)
    yn, bn, gn = W.to_oracle(y), W.to_oracle(b), W.to_oracle(g)
    x = (y.float() + b.float()).double().numpy()
    assert np.array_equal(O.bias_gelu_fwd(yn, bn), O.gelu_tanh(x))
    assert np.array_equal(O.bias_gelu_bwd(gn, yn, bn), O.gelu_tanh_grad(x) * g.double().numpy())


def _half_split(rows, F, first, second, dtype=torch.float32):
    return torch.cat([first, second], dim=1).to(dtype)


def test_geglu_with_unit_linear_half_is_gelu():
    """g2 = 1 makes GEGLU the bias-GeLU forward of the first half (catches
    activating the wrong half)."""
    rows, F = 3, 5
    a = torch.randn(rows, F)
    x = _half_split(rows, F, a, torch.ones(rows, F))
    out = O.bias_geglu_fwd(W.to_oracle(x))
    assert np.array_equal(out, O.bias_gelu_fwd(W.to_oracle(a)))
    zero = O.bias_geglu_fwd(W.to_oracle(_half_split(rows, F, a, torch.zeros(rows, F))))
    assert np.all(zero == 0)


def test_geglu_bias_is_added_before_split():
    rows, F = 2, 4
    x = torch.randn(rows, 2 * F)
    b = torch.randn(2 * F) * 0.5
    pre = (x + b).contiguous()   # fp32 add, exactly the bias add the op does
    assert np.array_equal(O.bias_geglu_fwd(W.to_oracle(x), W.to_oracle(b)),
                          O.bias_geglu_fwd(W.to_oracle(pre)))


def test_swiglu_with_unit_linear_half_is_silu():
    rows, F = 3, 7
    a = torch.randn(rows, F) * 3
    x = _half_split(rows, F, a, torch.ones(rows, F))
    out = O.bias_swiglu_fwd(W.to_oracle(x))
    ad = a.double().numpy()
    assert np.allclose(out, ad * expit(ad), rtol=4 * np.finfo(np.float64).eps, atol=0)
    x0 = _half_split(rows, F, torch.zeros(rows, F), torch.randn(rows, F))
    assert np.all(O.bias_swiglu_fwd(W.to_oracle(x0)) == 0)


def test_weighted_swiglu_identity():
    """weighted(x, w) == swiglu(x) * w, the identity the page's weighted-SwiGLU
    test checks (fusions page §9)."""
    x, b, g, w = W.glu_inputs(6, 11, torch.bfloat16, seed=5, with_weight=True)
    xn, bn, wn = W.to_oracle(x), W.to_oracle(b), W.to_oracle(w)
    plain = O.bias_swiglu_fwd(xn, bn)
    weighted = O.bias_swiglu_fwd(xn, bn, wn)
    assert np.allclose(weighted, plain * wn.astype(np.float64)[:, None], rtol=1e-15, atol=0)


def _dyadic(shape, seed, scale=4.0):
    """fp32 values on a 2^-10 grid so x +/- 2^-10 stays exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    return (torch.round(torch.randn(shape, generator=g) * scale * 1024) / 1024).float()


@pytest.mark.parametrize("op", ["geglu", "swiglu", "swiglu_w"])
def test_glu_backward_is_vjp_of_forward(op):
    """dx (and dweight) equal central differences of sum(g * forward)."""
    rows, F = 2, 3
    x = _dyadic((rows, 2 * F), 1, scale=2.0)
    g = torch.randn(rows, F, generator=torch.Generator().manual_seed(2))
    w = torch.rand(rows, generator=torch.Generator().manual_seed(3)) if op == "swiglu_w" else None
    xn, gn = W.to_oracle(x), W.to_oracle(g)
    wn = W.to_oracle(w)
    if op == "geglu":
        dx = O.bias_geglu_bwd(gn, xn)
        fwd = lambda xx, ww=None: O.bias_geglu_fwd(xx)
    else:
        dx, dw, _ = O.bias_swiglu_bwd(gn, xn, weight=wn)
        fwd = lambda xx, ww=wn: O.bias_swiglu_fwd(xx, weight=ww)
    gd = gn.astype(np.float64)
    h = 2.0 ** -10
    for i in range(rows):
        for j in range(2 * F):
            xp, xm = xn.copy(), xn.copy()
            xp[i, j] += np.float32(h)
            xm[i, j] -= np.float32(h)
            fd = ((gd * fwd(xp)).sum() - (gd * fwd(xm)).sum()) / (2 * h)
            assert abs(dx[i, j] - fd) <= 2e-5 * max(1.0, abs(fd)), (op, i, j, dx[i, j], fd)
    if op == "swiglu_w":
        for i in range(rows):
            wp, wm = wn.copy(), wn.copy()
            hw = 2.0 ** -12
            wp[i] += np.float32(hw)
            wm[i] -= np.float32(hw)
            fd = ((gd * fwd(xn, wp)).sum() - (gd * fwd(xn, wm)).sum()) / (2 * hw)
            assert abs(dw[i] - fd) <= 1e-9 * max(1.0, abs(fd))


def test_swiglu_dweight_abs_bounds_dweight():
    x, b, g, w = W.glu_inputs(5, 33, torch.bfloat16, seed=9, with_weight=True)
    _, dw, dwa = O.bias_swiglu_bwd(W.to_oracle(g), W.to_oracle(x), W.to_oracle(b), W.to_oracle(w))
    assert np.all(np.abs(dw) <= dwa) and np.all(dwa > 0)


# --------------------------------------------------------------------------
# bias-dropout-add (fusions page §3.2-§3.3)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("xdt,rdt", [(torch.bfloat16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                     (torch.float32, torch.float32), (torch.float32, torch.bfloat16)])
def test_dropout_inference_equals_torch_fp32_arithmetic(xdt, rdt):
    """In-place inference is (x + b) + residual.to(x.dtype) in fp32, bit for
    bit against torch's CPU fp32 ops (catches a missing cast of the residual,
    a wrong rounding order, or a dropped bias)."""
    x, b, r = W.dropout_inputs(7, 45, xdt, rdt, seed=21)
    ref = ((x.float() + b.float()) + r.to(xdt).float()).to(xdt)
    xn = W.to_oracle(x)
    O.bias_dropout_add_inference(xn, W.to_oracle(r), W.to_oracle(b))
    assert np.array_equal(xn, W.to_oracle(ref))


@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("xdt,rdt", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32)])
def test_dropout_train_equals_torch_given_mask(p, xdt, rdt):
    """Given the oracle's mask, out = (keep ? (x + b) * (1/(1-p)) : 0) + r~ is
    reproduced bit for bit by torch fp32 ops; dropped elements give exactly the
    cast residual."""
    x, b, r = W.dropout_inputs(9, 64, xdt, rdt, seed=4)
    out, keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b),
                                         p=p, seed=1234, offset=0)
    k = torch.from_numpy(keep.astype(bool))
    scale = torch.tensor(1.0, dtype=torch.float32) / (torch.tensor(1.0) - torch.tensor(p, dtype=torch.float32))
    v = x.float() + b.float()
    v = torch.where(k, v * scale, torch.zeros_like(v))
    rt = r.to(xdt).float()
    ref = (v + rt).to(xdt)
    assert np.array_equal(out, W.to_oracle(ref))
    dropped = ~k
    assert np.array_equal(W.to_oracle(ref)[dropped.numpy()], W.to_oracle(r.to(xdt))[dropped.numpy()])
    if p == 0.0:
        assert keep.all()


def test_dropout_threshold_definition():
    """keep iff u16 >= ceil(p * 65536), clamped to 65535."""
    for p in [0.0, 0.1, 0.25, 0.5, 0.9, 0.99999]:
        expect = min(65535, math.ceil(float(np.float32(p)) * 65536))
        assert O.dropout_threshold(p) == expect


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction_within_4_sigma(p):
    n = 1 << 20
    keep = O.keep_mask(1234, 0, 0, n, p)
    q = 1 - O.dropout_threshold(p) / 65536.0
    sigma = math.sqrt(q * (1 - q) / n)
    assert abs(keep.mean() - (1 - p)) <= 4 * sigma + 2e-5


def test_uniform16_histogram_chi_square():
    """The 16-bit words are uniform: chi-square over 256 buckets of the high
    byte and of the low byte (catches a biased lane mapping)."""
    from scipy.stats import chisquare
    n = 1 << 18
    keep_bits = np.array([O.uniform16(99, 3, e) for e in range(n)], dtype=np.uint32)
    for part in (keep_bits >> 8, keep_bits & 0xFF):
        counts = np.bincount(part.astype(np.int64), minlength=256)
        assert chisquare(counts).pvalue > 1e-4


def test_mask_sharding_invariance():
    """Two calls with elem_base = 0 and n/2 equal one call over n (the mask is
    a pure function of the global element index)."""
    n = 4096 + 24
    full = O.keep_mask(5, 7, 0, n, 0.3)
    half = n // 2 + 3  # not a multiple of 8: exercises a split inside a block
    assert np.array_equal(full, np.concatenate([O.keep_mask(5, 7, 0, half, 0.3),
                                                O.keep_mask(5, 7, half, n - half, 0.3)]))


def test_mask_depends_on_seed_and_offset():
    n = 1 << 16
    base = O.keep_mask(1234, 0, 0, n, 0.5)
    for other in (O.keep_mask(1235, 0, 0, n, 0.5), O.keep_mask(1234, 1, 0, n, 0.5),
                  O.keep_mask(1234 + (1 << 32), 0, 0, n, 0.5), O.keep_mask(1234, 1 << 32, 0, n, 0.5)):
        frac = (base != other).mean()
        assert abs(frac - 0.5) < 4 * math.sqrt(0.25 / n)


def test_dropout_train_mask_matches_keep_mask():
    x, b, r = W.dropout_inputs(5, 40, torch.bfloat16, torch.float32, seed=2)
    _, keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=0.5,
                                       seed=77, offset=9, elem_base=123)
    assert np.array_equal(keep.ravel(), O.keep_mask(77, 9, 123, 200, 0.5))


def test_uniform16_is_the_little_endian_word_of_the_block():
    """Element e reads 16-bit word e % 8 of the 128-bit Philox4x32-10 block
    e / 8 seen as little-endian bytes, with counter (lo j, hi j, lo offset,
    hi offset) and key (lo seed, hi seed).  Formulated with a byte view of the
    block, not with shifts, so a permuted lane or counter layout fails."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        offset = int(rng.integers(0, 2**64, dtype=np.uint64))
        e = int(rng.integers(0, 2**40))
        j = e // 8
        ctr = np.array([j & 0xFFFFFFFF, j >> 32, offset & 0xFFFFFFFF, offset >> 32], dtype=np.uint32)
        key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
        block = O.philox4x32_10(ctr, key).astype("<u4")
        assert O.uniform16(seed, offset, e) == int(block.view("<u2")[e % 8])


def test_condition_scales_bound_the_derivatives():
    """The backward ops' condition scale is |sum of terms| <= sum |terms|:
    never below |value|, equal to it where no term is negative (gelu' for
    x >= 0, silu' for a >= 0), and far above it at the derivative's root."""
    y = torch.linspace(-6, 6, 4801).reshape(1, -1)
    g = torch.ones_like(y)
    dy, sc = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), with_scale=True)
    assert np.all(sc >= np.abs(dy) * (1 - 1e-15))
    pos = y.numpy() >= 0
    assert np.allclose(sc[pos], np.abs(dy[pos]), rtol=1e-14, atol=0)
    root = np.abs(y.numpy() + 0.7518) < 2e-3
    assert np.all(sc[root] > 100 * np.abs(dy[root]))
    F = y.shape[1]
    x = torch.cat([y, torch.ones_like(y)], dim=1)
    dx, _, _, sx = O.bias_swiglu_bwd(W.to_oracle(g), W.to_oracle(x), with_scale=True)
    assert np.all(sx >= np.abs(dx) * (1 - 1e-15))
    assert np.allclose(sx[:, :F][pos], np.abs(dx[:, :F][pos]), rtol=1e-14, atol=0)
    dg, sg = O.bias_geglu_bwd(W.to_oracle(g), W.to_oracle(x), with_scale=True)
    assert np.all(sg >= np.abs(dg) * (1 - 1e-15))



# --------------------------------------------------------------------------
# bias-dropout-add backward and the bias gradient (column sums)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("xdt,rdt", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32),
                                     (torch.bfloat16, torch.bfloat16)])
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_dropout_backward_equals_torch_given_mask(xdt, rdt, p):
    """dx = keep ? g * (1/(1-p)) : 0 and dres = g.to(residual dtype), bit for
    bit against torch fp32 ops; the regenerated mask equals the forward's."""
    x, b, r = W.dropout_inputs(6, 72, xdt, rdt, seed=13)
    g = W.normal((6, 72), xdt, 14)
    _, keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=p,
                                       seed=55, offset=3, elem_base=17)
    rname = "bf16" if rdt == torch.bfloat16 else "f32"
    dx, dres = O.bias_dropout_add_bwd(W.to_oracle(g), keep, p=p, res_dtype=rname)
    dx2, _ = O.bias_dropout_add_bwd(W.to_oracle(g), None, p=p, seed=55, offset=3, elem_base=17)
    assert np.array_equal(dx, dx2)
    scale = torch.tensor(1.0, dtype=torch.float32) / (torch.tensor(1.0) - torch.tensor(p, dtype=torch.float32))
    k = torch.from_numpy(keep.astype(bool))
    ref = torch.where(k, g.float() * scale, torch.zeros(6, 72)).to(xdt)
    assert np.array_equal(dx, W.to_oracle(ref))
    assert np.array_equal(dres, W.to_oracle(g.to(rdt)))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_column_sums_are_sums_of_stored_values(dt):
    """The bias gradient sums the gradient as stored (rounded to its dtype),
    checked against torch's float64 sum of the rounded tensor."""
    v = torch.randn(37, 19, dtype=torch.float64) * 3
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    stored = v.float().to(tdt).double()
    s, a = O.column_sums(v.numpy(), dt)
    assert np.allclose(s, stored.sum(0).numpy(), rtol=1e-14, atol=1e-12)
    assert np.allclose(a, stored.abs().sum(0).numpy(), rtol=1e-14, atol=1e-12)



# --------------------------------------------------------------------------
# weighted squared ReLU
# --------------------------------------------------------------------------
def test_weighted_squared_relu_matches_torch_float64():
    """relu(x)^2 * w against torch's own float64 relu, square and product."""
    x = W.normal((7, 33), torch.bfloat16, 61)
    w = W.uniform((7,), 62)
    out = O.weighted_squared_relu_fwd(W.to_oracle(x), W.to_oracle(w))
    ref = torch.relu(x.double()) ** 2 * w.double()[:, None]
    assert np.allclose(out, ref.numpy(), rtol=1e-15, atol=0)
    assert np.all(out[x.float().numpy() <= 0] == 0)


def test_weighted_squared_relu_backward_is_vjp():
    """dx and dweight equal central differences of sum(g * forward)."""
    rows, cols = 3, 5
    x = _dyadic((rows, cols), 5, scale=2.0)
    g = torch.randn(rows, cols, generator=torch.Generator().manual_seed(6))
    w = torch.rand(rows, generator=torch.Generator().manual_seed(7))
    xn, gn, wn = W.to_oracle(x), W.to_oracle(g), W.to_oracle(w)
    dx, dw, dwa = O.weighted_squared_relu_bwd(gn, xn, wn)
    gd = gn.astype(np.float64)
    h = 2.0 ** -10
    for i in range(rows):
        for j in range(cols):
            if abs(xn[i, j]) <= h:       # relu is not differentiable at 0
                continue
            xp, xm = xn.copy(), xn.copy()
            xp[i, j] += np.float32(h)
            xm[i, j] -= np.float32(h)
            fd = ((gd * O.weighted_squared_relu_fwd(xp, wn)).sum() -
                  (gd * O.weighted_squared_relu_fwd(xm, wn)).sum()) / (2 * h)
            assert abs(dx[i, j] - fd) <= 1e-9 * max(1.0, abs(fd))
        wp, wm = wn.copy(), wn.copy()
        wp[i] += np.float32(2.0 ** -12)
        wm[i] -= np.float32(2.0 ** -12)
        fd = ((gd * O.weighted_squared_relu_fwd(xn, wp)).sum() -
              (gd * O.weighted_squared_relu_fwd(xn, wm)).sum()) / (2 * 2.0 ** -12)
        assert abs(dw[i] - fd) <= 1e-9 * max(1.0, abs(fd))
    assert np.all(np.abs(dw) <= dwa)
