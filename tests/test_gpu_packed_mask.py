"""The bit-packed keep mask of bias-dropout-add (mfx_bias_dropout_add_train_packed
and mfx_bias_dropout_add_bwd_packed): one bit per element, element i at bit
i % 8 of byte i // 8.  The packed mask must be the oracle's byte mask packed
by numpy (np.packbits, least significant bit first), the outputs the
oracle's bits, and both equal to the byte-mask calls'; the backward from the
bits must equal the backward from the bytes.  Ragged sizes (the last byte
partial, spans whose mask is not a whole number of 16-byte copies), element
offsets (the element-wise path) and the D2 layer shape are covered."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def on(t):
    return None if t is None else t.to(DEV)


def at_offset(t, k):
    t = t.to(DEV)
    buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[k:k + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def packbits(keep):
    return np.packbits(np.asarray(keep, dtype=np.uint8).ravel(), bitorder="little")


SHAPES = [(1, 1), (1, 7), (2, 9), (3, 4099), (5, 24), (16, 4096), (7, 13), (33, 1023), (300, 4104)]


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (BF16, BF16), (F32, F32), (F32, BF16)])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("elem_base", [0, 5])
def test_packed_train_bit_exact(xdt, rdt, shape, p, elem_base):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows * 13 + cols)
    seed, offset = 1234, 7
    ref_out, ref_keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=p, seed=seed,
                                                 offset=offset, elem_base=elem_base)
    out, kb = mfx.mfx_bias_dropout_add_train_packed(on(x), on(b), on(r), p, seed, offset, elem_base)
    out8, keep8 = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), p, seed, offset, elem_base)
    torch.cuda.synchronize()
    assert np.array_equal(kb.cpu().numpy(), packbits(ref_keep))
    assert np.array_equal(W.to_oracle(out), ref_out)
    assert np.array_equal(bits(out), bits(out8)) and np.array_equal(kb.cpu().numpy(), packbits(keep8.cpu()))


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (BF16, BF16), (F32, F32)])
@pytest.mark.parametrize("k", [1, 3])
def test_packed_train_misaligned(xdt, rdt, k):
    """Data one or three elements off a 16-byte boundary: the element-wise
    path, same bits."""
    rows, cols = 37, 1030
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=k)
    ref_out, ref_keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=0.3, seed=9,
                                                 offset=2, elem_base=11)
    out = at_offset(torch.zeros(rows, cols, dtype=xdt), k)
    kb = at_offset(torch.zeros((rows * cols + 7) // 8, dtype=torch.uint8), k)
    mfx.mfx_bias_dropout_add_train_packed(at_offset(x, k), at_offset(b, k), at_offset(r, k), 0.3, 9, 2, 11,
                                          out=out, keep_bits=kb)
    torch.cuda.synchronize()
    assert np.array_equal(kb.cpu().numpy(), packbits(ref_keep))
    assert np.array_equal(W.to_oracle(out), ref_out)


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (BF16, BF16), (F32, F32), (F32, BF16)])
@pytest.mark.parametrize("shape", SHAPES + [(1, 4111), (64, 4100)])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_packed_bwd_bit_exact(xdt, rdt, shape, p):
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + 3 * cols)
    g = W.normal((rows, cols), xdt, 41)
    _, kb = mfx.mfx_bias_dropout_add_train_packed(on(x), on(b), on(r), p, 77, 3)
    _, keep8 = mfx.mfx_bias_dropout_add_train(on(x), on(b), on(r), p, 77, 3)
    dx, dres = mfx.mfx_bias_dropout_add_bwd_packed(on(g), kb, p, residual_dtype=rdt)
    dx8, dres8 = mfx.mfx_bias_dropout_add_bwd(on(g), keep8, p, residual_dtype=rdt)
    torch.cuda.synchronize()
    ref_dx, ref_dres = O.bias_dropout_add_bwd(W.to_oracle(g), keep8.cpu().numpy(), p=p,
                                              res_dtype="bf16" if rdt == BF16 else "f32")
    assert np.array_equal(W.to_oracle(dx), ref_dx)
    assert np.array_equal(bits(dx), bits(dx8))
    if rdt != xdt:
        assert np.array_equal(W.to_oracle(dres), ref_dres) and np.array_equal(bits(dres), bits(dres8))
    # the bits misaligned (element-wise path) give the same result
    kbm = at_offset(kb, 1)
    dxm, _ = mfx.mfx_bias_dropout_add_bwd_packed(on(g), kbm, p)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dxm), bits(dx))


def test_packed_full_size_d2():
    """[4096 x 4] x 4096, bf16 x, fp32 residual, p = 0.1, seed 1234: the bits
    are the byte mask's, training and backward outputs the same bits."""
    x, b, r = W.dropout_inputs(16384, 4096, BF16, F32, seed=0, device=DEV)
    g = W.normal((16384, 4096), BF16, 5, device=DEV)
    out, kb = mfx.mfx_bias_dropout_add_train_packed(x, b, r, 0.1, 1234, 0)
    out8, keep8 = mfx.mfx_bias_dropout_add_train(x, b, r, 0.1, 1234, 0)
    dx, dres = mfx.mfx_bias_dropout_add_bwd_packed(g, kb, 0.1, residual_dtype=F32)
    dx8, dres8 = mfx.mfx_bias_dropout_add_bwd(g, keep8, 0.1, residual_dtype=F32)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out8.view(torch.int16))
    assert np.array_equal(kb.cpu().numpy(), packbits(keep8.cpu().numpy()))
    assert torch.equal(dx.view(torch.int16), dx8.view(torch.int16)) and torch.equal(dres, dres8)
    kept = float(keep8.float().mean())
    n = keep8.numel()
    assert abs(kept - (1 - np.ceil(0.1 * 65536) / 65536)) < 4 * np.sqrt(0.1 * 0.9 / n)
    assert mfx.mfx_device_error() == 0
