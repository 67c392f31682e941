"""Comparison rules between the CUDA path and the oracle.

bf16 outputs: within 1 bf16 ulp of the oracle's unrounded value, the ulp taken
at the oracle value's binade (2^(e - 7) for |ref| in [2^e, 2^(e+1)), and the
smallest subnormal step 2^-133 below the normal range), so either bf16
neighbour of the reference passes.

fp32 outputs: max absolute error 1e-6 against the oracle.  Where |ref| >= 4
one fp32 ulp is already 4.8e-7 (9.5e-7 from 8), so 1e-6 is two ulps or less
there; for those elements the rule is a distance of at most 2 fp32 ulps at
the reference's binade.  This reading of the 1e-6 gate is written out here
and nowhere loosened.

Derivatives that cross zero: the backward ops form their factor as a sum of
terms that cancel at its root (gelu' near x = -0.75, silu' near a = -1.278).
There the fp32 result carries rounding error relative to the magnitude of
the terms, not of the result, so both rules above add 16 * 2^-24 * scale,
where `scale` is the oracle's per-element magnitude of those terms times the
other factors.  Away from the roots scale ~ |ref| and the term is below 1/2000
of a bf16 ulp.

Integer/byte outputs (dropout masks) and the dropout values: bit-exact.
"""
import numpy as np
import torch


def to_f64(t):
    """A torch tensor (any float dtype, any device) as a float64 numpy array."""
    return t.detach().float().cpu().double().numpy()


def _binade_ulp(ref, mant_bits, min_exp):
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, min_exp), min_exp)
    return np.exp2(e - mant_bits)


def bf16_ulp(ref):
    return _binade_ulp(ref, 7, -126)


def f32_ulp(ref):
    return _binade_ulp(ref, 23, -126)


# Smallest magnitude that rounds to infinity (round-to-nearest) in each format.
BF16_OVERFLOW = (2.0 - 2.0 ** -8) * 2.0 ** 127
F32_OVERFLOW = (2.0 - 2.0 ** -24) * 2.0 ** 127


def _saturate(ref, limit):
    """The oracle's fp64 value as the output format must hold it: values at
    or past the rounding threshold become infinities."""
    return np.where(np.abs(ref) >= limit, np.copysign(np.inf, ref), ref)


def _special(got, ref):
    """Positions where either side is NaN/inf must agree exactly in kind."""
    bad = np.isnan(got) != np.isnan(ref)
    inf = np.isinf(ref) | np.isinf(got)
    bad |= inf & ~np.isnan(ref) & (got != ref)
    return bad, np.isnan(ref) | inf


COND_UNITS = 16 * 2.0 ** -24


def check_bf16(got, ref, what="", scale=None):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = _saturate(np.asarray(ref, dtype=np.float64), BF16_OVERFLOW)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bad, skip = _special(got, ref)
    err = np.where(skip, 0.0, np.abs(got - ref))
    tol = bf16_ulp(ref)
    if scale is not None:
        tol = tol + COND_UNITS * np.asarray(scale, dtype=np.float64)
    ratio = err / tol
    bad |= ratio > 1.0
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} bf16 outputs beyond 1 ulp; "
                             f"max ratio {ratio.max():.3f}; first at flat {i}: got "
                             f"{got.ravel()[i]} ref {ref.ravel()[i]}")
    return float(ratio.max()) if ratio.size else 0.0


def check_f32(got, ref, what="", scale=None):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = _saturate(np.asarray(ref, dtype=np.float64), F32_OVERFLOW)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bad, skip = _special(got, ref)
    err = np.where(skip, 0.0, np.abs(got - ref))
    big = np.abs(ref) >= 4.0
    cond = 0.0 if scale is None else COND_UNITS * np.asarray(scale, dtype=np.float64)
    ulps = np.maximum(err - cond, 0.0) / f32_ulp(ref)
    bad |= np.where(big, ulps > 2.0, err > 1e-6 + cond)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} fp32 outputs out of tolerance; "
                             f"max abs {err.max():.3e}, max ulps {ulps.max():.2f}; first at flat "
                             f"{i}: got {got.ravel()[i]} ref {ref.ravel()[i]}")
    small = ~big
    return (float(err[small].max()) if small.any() else 0.0,
            float(ulps[big].max()) if big.any() else 0.0)


def check(got, ref, what="", scale=None):
    if got.dtype == torch.bfloat16:
        return check_bf16(got, ref, what, scale)
    return check_f32(got, ref, what, scale)


def bits(t):
    """Raw bit patterns of a tensor (for bit-exact comparisons)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()
