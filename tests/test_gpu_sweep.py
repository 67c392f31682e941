"""Parity over the sweep of workload shapes: tokens {512, 4096, 32768, 65536}
x hidden {1024, 4096, 4099, 8192, 16384} (4099 exercises the tails), every
op, bf16 and fp32, dropout p in {0, 0.1, 0.5}, residual in x's dtype plus the
fp32-residual case for bf16.  Each op runs on the whole tensor in the launch
configuration the library picks for that size; whole sampled rows are
compared with the oracle (dropout rows with their own elem_base, so masks are
checked bit for bit)."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bits, check

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda"
BF16, F32 = torch.bfloat16, torch.float32
SHAPES = [(t, h) for t in W.SWEEP_TOKENS for h in W.SWEEP_HIDDEN]


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()
    yield
    torch.cuda.empty_cache()


def rows_of(T, k=3, seed=0):
    g = np.random.default_rng(seed + T)
    return sorted(set(g.choice(T, k, replace=False).tolist()) | {T - 1})


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("T,H", SHAPES)
def test_sweep_gelu(dtype, T, H):
    y, b, g = W.gelu_inputs(T, H, dtype, seed=T + H, device=DEV)
    out = mfx.mfx_bias_gelu_fwd(b, y)
    dy = mfx.mfx_bias_gelu_bwd(g, b, y)
    torch.cuda.synchronize()
    rows = rows_of(T)
    yo, go, bo = W.to_oracle(y[rows]), W.to_oracle(g[rows]), W.to_oracle(b)
    check(out[rows], O.bias_gelu_fwd(yo, bo), f"sweep gelu fwd {dtype} {T}x{H}")
    ref, sc = O.bias_gelu_bwd(go, yo, bo, with_scale=True)
    check(dy[rows], ref, f"sweep gelu bwd {dtype} {T}x{H}", sc)
    del y, g, out, dy


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("T,F", SHAPES)
@pytest.mark.parametrize("kind", ["geglu", "swiglu_w"])
def test_sweep_glu(kind, dtype, T, F):
    x, b, g, w = W.glu_inputs(T, F, dtype, seed=T + F, device=DEV, with_weight=kind == "swiglu_w")
    if kind == "geglu":
        f = mfx.mfx_bias_geglu_fwd(x, b)
        dx = mfx.mfx_bias_geglu_bwd(g, x, b)
        dw = None
    else:
        f = mfx.mfx_bias_swiglu_fwd(x, b, w)
        dx, dw = mfx.mfx_bias_swiglu_bwd(g, x, b, w)
    torch.cuda.synchronize()
    rows = rows_of(T, seed=1)
    xo, go, bo = W.to_oracle(x[rows]), W.to_oracle(g[rows]), W.to_oracle(b)
    if kind == "geglu":
        check(f[rows], O.bias_geglu_fwd(xo, bo), f"sweep geglu fwd {dtype} {T}x{F}")
        ref, sc = O.bias_geglu_bwd(go, xo, bo, with_scale=True)
        check(dx[rows], ref, f"sweep geglu bwd {dtype} {T}x{F}", sc)
    else:
        wo = W.to_oracle(w[rows])
        check(f[rows], O.bias_swiglu_fwd(xo, bo, wo), f"sweep swiglu_w fwd {dtype} {T}x{F}")
        ref, rdw, rdwa, sc = O.bias_swiglu_bwd(go, xo, bo, wo, with_scale=True)
        check(dx[rows], ref, f"sweep swiglu_w bwd {dtype} {T}x{F}", sc)
        err = np.abs(dw[rows].double().cpu().numpy() - rdw)
        assert np.all(err <= 1e-5 * rdwa)
    del x, g, f, dx


@pytest.mark.parametrize("xdt,rdt", [(BF16, BF16), (BF16, F32), (F32, F32)])
@pytest.mark.parametrize("T,H", SHAPES)
def test_sweep_dropout(xdt, rdt, T, H):
    x, b, r = W.dropout_inputs(T, H, xdt, rdt, seed=T * 7 + H, device=DEV)
    rows = rows_of(T, seed=2)
    x_rows = W.to_oracle(x[rows])
    for p in W.SWEEP_P:
        out, keep = mfx.mfx_bias_dropout_add_train(x, b, r, p, 1234, 0)
        torch.cuda.synchronize()
        for row in rows:
            ro, rk = O.bias_dropout_add_train(W.to_oracle(x[row:row + 1]), W.to_oracle(r[row:row + 1]),
                                              W.to_oracle(b), p=p, seed=1234, offset=0,
                                              elem_base=row * H)
            assert np.array_equal(keep[row:row + 1].cpu().numpy(), rk), (p, row)
            assert np.array_equal(bits(out[row:row + 1]), ro.view(bits(out).dtype)), (p, row)
        del out, keep
    mfx.mfx_bias_dropout_add_inference(x, b, r)
    torch.cuda.synchronize()
    O.bias_dropout_add_inference(x_rows, W.to_oracle(r[rows]), W.to_oracle(b))
    assert np.array_equal(bits(x[rows]), x_rows.view(bits(x).dtype))
    assert mfx.mfx_device_error() == 0
