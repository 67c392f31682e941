"""Parity at the full workload sizes, with the launch configuration the
benchmark times: every element where the oracle is fast enough (the fp32
1024x4096 case), sampled whole rows elsewhere, and whole-tensor properties
(mask statistics, exact dropout arithmetic against torch's own fp32 ops)."""
import math

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
N_SAMPLE_ROWS = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def sample_rows(rows, seed=0):
    g = np.random.default_rng(seed)
    pick = set(g.choice(rows, N_SAMPLE_ROWS - 3, replace=False).tolist()) | {0, rows // 2, rows - 1}
    return sorted(pick)


def test_gelu_fp32_1024x4096_every_element():
    wl = W.GELU_F32_SMALL
    y, b, g = W.gelu_inputs(wl.rows, wl.width, wl.dtype, seed=0, device=DEV)
    out = mfx.mfx_bias_gelu_fwd(b, y)
    dy = mfx.mfx_bias_gelu_bwd(g, b, y)
    torch.cuda.synchronize()
    yo, bo, go = W.to_oracle(y), W.to_oracle(b), W.to_oracle(g)
    check(out, O.bias_gelu_fwd(yo, bo), "gelu fp32 fwd full")
    ref, sc = O.bias_gelu_bwd(go, yo, bo, with_scale=True)
    check(dy, ref, "gelu fp32 bwd full", sc)


def test_gelu_bf16_16384x16384_sampled_rows():
    wl = W.GELU_BF16
    y, b, g = W.gelu_inputs(wl.rows, wl.width, wl.dtype, seed=0, device=DEV)
    out = mfx.mfx_bias_gelu_fwd(b, y)
    dy = mfx.mfx_bias_gelu_bwd(g, b, y)
    torch.cuda.synchronize()
    rows = sample_rows(wl.rows)
    bo = W.to_oracle(b)
    yo, go = W.to_oracle(y[rows]), W.to_oracle(g[rows])
    check(out[rows], O.bias_gelu_fwd(yo, bo), "gelu bf16 fwd sampled")
    ref, sc = O.bias_gelu_bwd(go, yo, bo, with_scale=True)
    check(dy[rows], ref, "gelu bf16 bwd sampled", sc)
    assert torch.isfinite(out.float()).all() and torch.isfinite(dy.float()).all()


@pytest.mark.parametrize("kind", ["geglu", "swiglu", "swiglu_w"])
def test_glu_bf16_16384x28672_sampled_rows(kind):
    wl = W.GLU_BF16
    x, b, g, w = W.glu_inputs(wl.rows, wl.width, wl.dtype, seed=0, device=DEV,
                              with_weight=kind == "swiglu_w")
    dw = None
    if kind == "geglu":
        f = mfx.mfx_bias_geglu_fwd(x, b)
        dx = mfx.mfx_bias_geglu_bwd(g, x, b)
    else:
        f = mfx.mfx_bias_swiglu_fwd(x, b, w)
        dx, dw = mfx.mfx_bias_swiglu_bwd(g, x, b, w)
    torch.cuda.synchronize()
    rows = sample_rows(wl.rows, seed=1)
    xo, go, bo = W.to_oracle(x[rows]), W.to_oracle(g[rows]), W.to_oracle(b)
    if kind == "geglu":
        check(f[rows], O.bias_geglu_fwd(xo, bo), "geglu fwd sampled")
        ref, sc = O.bias_geglu_bwd(go, xo, bo, with_scale=True)
        check(dx[rows], ref, "geglu bwd sampled", sc)
    else:
        wo = W.to_oracle(w[rows]) if w is not None else None
        check(f[rows], O.bias_swiglu_fwd(xo, bo, wo), f"{kind} fwd sampled")
        rdx, rdw, rdwa, sc = O.bias_swiglu_bwd(go, xo, bo, wo, with_scale=True)
        check(dx[rows], rdx, f"{kind} bwd sampled", sc)
        if w is not None:
            err = np.abs(dw[rows].double().cpu().numpy() - rdw)
            assert np.all(err <= 1e-5 * rdwa)


def test_dropout_bf16_fp32_residual_full_size():
    wl = W.DROPOUT_BF16
    x, b, r = W.dropout_inputs(wl.rows, wl.width, wl.dtype, wl.residual_dtype, seed=0, device=DEV)
    out, keep = mfx.mfx_bias_dropout_add_train(x, b, r, wl.p, wl.dropout_seed, wl.dropout_offset)
    torch.cuda.synchronize()
    # kept fraction over all 67M elements within 4 sigma of the keep probability
    n = keep.numel()
    q = 1 - O.dropout_threshold(wl.p) / 65536
    frac = keep.double().mean().item()
    assert abs(frac - q) <= 4 * math.sqrt(q * (1 - q) / n)
    assert abs(frac - (1 - wl.p)) <= 4 * math.sqrt(wl.p * (1 - wl.p) / n) + 1e-5
    # whole tensor against torch's own fp32 ops given the mask
    scale = torch.tensor(1.0, dtype=torch.float32) / (torch.tensor(1.0) - torch.tensor(wl.p, dtype=torch.float32))
    v = x.float() + b.float()
    v = torch.where(keep.bool(), v * scale.to(DEV), torch.zeros_like(v))
    ref = (v + r.to(wl.dtype).float()).to(wl.dtype)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # sampled rows against the oracle, mask included (elem_base = row * cols)
    for row in sample_rows(wl.rows, seed=2):
        ro, rk = O.bias_dropout_add_train(W.to_oracle(x[row:row + 1]), W.to_oracle(r[row:row + 1]),
                                          W.to_oracle(b), p=wl.p, seed=wl.dropout_seed,
                                          offset=wl.dropout_offset, elem_base=row * wl.width)
        assert np.array_equal(keep[row:row + 1].cpu().numpy(), rk)
        assert np.array_equal(bits(out[row:row + 1]), ro.view(np.int16))


def test_dropout_inference_full_size_in_place():
    wl = W.DROPOUT_BF16
    x, b, r = W.dropout_inputs(wl.rows, wl.width, wl.dtype, wl.residual_dtype, seed=0, device=DEV)
    ref = ((x.float() + b.float()) + r.to(wl.dtype).float()).to(wl.dtype)
    rows = sample_rows(wl.rows, seed=3)
    x_rows = W.to_oracle(x[rows])
    ptr = x.data_ptr()
    ret = mfx.mfx_bias_dropout_add_inference(x, b, r, wl.p, wl.dropout_seed, wl.dropout_offset)
    torch.cuda.synchronize()
    assert ret.data_ptr() == ptr
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
    O.bias_dropout_add_inference(x_rows, W.to_oracle(r[rows]), W.to_oracle(b))
    assert np.array_equal(bits(x[rows]), x_rows.view(np.int16))


@pytest.mark.parametrize("regen", [False, True])
def test_dropout_backward_full_size(regen):
    """Backward on the [4096*4 x 4096] workload: whole tensor against torch's
    fp32 ops given the forward's mask (bit-exact), sampled rows against the
    oracle with the mask regenerated."""
    wl = W.DROPOUT_BF16
    x, b, r = W.dropout_inputs(wl.rows, wl.width, wl.dtype, wl.residual_dtype, seed=0, device=DEV)
    g = W.normal((wl.rows, wl.width), wl.dtype, 5, device=DEV)
    _, keep = mfx.mfx_bias_dropout_add_train(x, b, r, wl.p, wl.dropout_seed, wl.dropout_offset)
    dx, dres = mfx.mfx_bias_dropout_add_bwd(g, None if regen else keep, wl.p, wl.dropout_seed,
                                            wl.dropout_offset, residual_dtype=torch.float32)
    torch.cuda.synchronize()
    scale = torch.tensor(1.0, dtype=torch.float32) / (torch.tensor(1.0) - torch.tensor(wl.p, dtype=torch.float32))
    ref = torch.where(keep.bool(), g.float() * scale.to(DEV), torch.zeros_like(g, dtype=torch.float32))
    assert torch.equal(dx.view(torch.int16), ref.to(wl.dtype).view(torch.int16))
    assert torch.equal(dres, g.float())
    for row in sample_rows(wl.rows, seed=4):
        rdx, _ = O.bias_dropout_add_bwd(W.to_oracle(g[row:row + 1]), None, p=wl.p, seed=wl.dropout_seed,
                                        offset=wl.dropout_offset, elem_base=row * wl.width)
        assert np.array_equal(bits(dx[row:row + 1]), rdx.view(np.int16))


def test_weighted_squared_relu_bf16_16384x14336_sampled_rows():
    wl = W.SQRELU_BF16
    x, g, w = W.sqrelu_inputs(wl.rows, wl.width, wl.dtype, seed=60, device=DEV)
    out = mfx.mfx_weighted_squared_relu_fwd(x, w)
    dx, dw = mfx.mfx_weighted_squared_relu_bwd(g, x, w)
    torch.cuda.synchronize()
    rows = sample_rows(wl.rows, seed=6)
    xo, go, wo = W.to_oracle(x[rows]), W.to_oracle(g[rows]), W.to_oracle(w[rows])
    check(out[rows], O.weighted_squared_relu_fwd(xo, wo), "sqrelu fwd sampled")
    rdx, rdw, rdwa = O.weighted_squared_relu_bwd(go, xo, wo)
    check(dx[rows], rdx, "sqrelu bwd sampled")
    err = np.abs(dw[rows].double().cpu().numpy() - rdw)
    assert np.all(err <= 1e-5 * rdwa + 1e-30)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_bf16_benchmark_size_sampled_rows(causal):
    """[2, 32, 4096, 4096] with a padding mask (or the causal form on
    [64, 4096, 4096]), the benchmark's launches, checked on sampled rows.
    The oracle takes each sampled row alone, with its mask row (the causal
    row q as the additive mask 0 up to q and -inf after, which the pins show
    equal to the causal form); the backward is fed the oracle's rounded
    forward on those rows."""
    b, heads, sq, sk = 2, 32, 4096, 4096
    x, m, dy, scale = W.softmax_inputs(b, heads, sq, sk, torch.bfloat16, seed=70, device=DEV,
                                       mask=None if causal else "pad")
    if causal:
        y = mfx.mfx_scaled_upper_triang_masked_softmax_fwd(x.view(b * heads, sq, sk), scale)
    else:
        y = mfx.mfx_scaled_masked_softmax_fwd(x, scale, m)
    torch.cuda.synchronize()
    fx, fy, fdy = (t.reshape(-1, sk) for t in (x, y, dy))
    rows = sample_rows(fx.shape[0], seed=7)

    def row_mask(r):
        if causal:
            q = r % sq
            mr = torch.zeros(sk)
            mr[q + 1:] = float("-inf")
            return mr.to(torch.bfloat16).reshape(1, 1, 1, sk)
        return m[r // (heads * sq)].reshape(1, 1, 1, sk).cpu()

    yin = fy.clone()
    for r in rows:
        ref = O.scaled_masked_softmax_fwd(W.to_oracle(fx[r].reshape(1, 1, 1, sk).cpu()), scale,
                                          mask=W.to_oracle(row_mask(r)))[0, 0, 0]
        check(fy[r].cpu(), ref, f"softmax fwd row {r}")
        yin[r] = torch.from_numpy(ref).to(torch.bfloat16).to(DEV)
    if causal:
        dx = mfx.mfx_scaled_upper_triang_masked_softmax_bwd(fdy.view(b * heads, sq, sk),
                                                             yin.view(b * heads, sq, sk), scale)
    else:
        dx = mfx.mfx_scaled_masked_softmax_bwd(fdy, yin, scale)
    torch.cuda.synchronize()
    fdx = dx.reshape(-1, sk)
    for r in rows:
        # excluded positions hold y = 0, so the row-alone backward is the causal one there too
        ref, sc = O.scaled_softmax_bwd(W.to_oracle(fdy[r].reshape(1, sk).cpu()),
                                       W.to_oracle(yin[r].reshape(1, sk).cpu()), scale, with_scale=True)
        check(fdx[r].cpu(), ref[0], f"softmax bwd row {r}", sc[0])
