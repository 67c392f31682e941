"""The pipelined kernels on any width and any common misalignment.

Bias-GeLU and bias-dropout-add stream 8-element units of the flat tensor
through the bulk-copy ring whenever every pointer sits the same whole number
of elements below a 16-byte boundary: those elements (the head) and the last
n mod 8 (the tail) are done one by one, and a unit stride that is a multiple
of cols / gcd(cols, 8) keeps each thread on one column phase for any width.
These tests pin that path to the oracle at odd widths and at every element
offset, check that it gives the same bits as the aligned path and the
element-wise path (pointers misaligned by different amounts), and cover
in-place calls and the dropout generator's block alignment (elem_base)."""
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
BF16, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


def at_offset(t, k):
    """A device copy of t whose data starts k elements past a 16-byte
    boundary (k = 0: aligned)."""
    t = t.to(DEV)
    buf = torch.zeros(t.numel() + 16, dtype=t.dtype, device=DEV)
    assert buf.data_ptr() % 16 == 0
    v = buf[k:k + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def empty_at(shape, dtype, k):
    return at_offset(torch.zeros(shape, dtype=dtype), k)


def offsets(dtype):
    return [0, 1, 2, 3, 5, 7] if dtype == BF16 else [0, 1, 2, 3]


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("shape", [(300, 4099), (129, 1023), (64, 5), (9, 3), (2, 4105), (40, 1032)])
def test_bias_gelu_any_width_every_offset(dtype, shape):
    rows, cols = shape
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=rows * 7 + cols)
    ref_f = O.bias_gelu_fwd(W.to_oracle(y), W.to_oracle(b))
    ref_b, scale_b = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b), with_scale=True)
    first = None
    for k in offsets(dtype):
        out = mfx.mfx_bias_gelu_fwd(at_offset(b, k), at_offset(y, k), out=empty_at(y.shape, dtype, k))
        dy = mfx.mfx_bias_gelu_bwd(at_offset(g, k), at_offset(b, k), at_offset(y, k),
                                   dy=empty_at(y.shape, dtype, k))
        torch.cuda.synchronize()
        check(out, ref_f, f"fwd offset {k}")
        check(dy, ref_b, f"bwd offset {k}", scale_b)
        if first is None:
            first = (bits(out), bits(dy))
        else:                                      # every offset gives the aligned bits
            assert np.array_equal(bits(out), first[0]) and np.array_equal(bits(dy), first[1]), k
    # pointers misaligned by different amounts take the element-wise path: same bits
    out_m = mfx.mfx_bias_gelu_fwd(at_offset(b, 3), at_offset(y, 1), out=empty_at(y.shape, dtype, 2))
    dy_m = mfx.mfx_bias_gelu_bwd(at_offset(g, 2), at_offset(b, 0), at_offset(y, 1), dy=empty_at(y.shape, dtype, 1))
    torch.cuda.synchronize()
    assert np.array_equal(bits(out_m), first[0]) and np.array_equal(bits(dy_m), first[1])
    assert mfx.mfx_device_error() == 0


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_bias_gelu_misaligned_in_place(dtype):
    rows, cols = 257, 4099
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=11)
    ref = mfx.mfx_bias_gelu_fwd(b.to(DEV), y.to(DEV))
    ref_b = mfx.mfx_bias_gelu_bwd(g.to(DEV), b.to(DEV), y.to(DEV))
    yk = at_offset(y, 3)
    mfx.mfx_bias_gelu_fwd(at_offset(b, 1), yk, out=yk)                 # out == y
    gk = at_offset(g, 3)
    mfx.mfx_bias_gelu_bwd(gk, at_offset(b, 0), at_offset(y, 3), dy=gk)  # dy == g
    torch.cuda.synchronize()
    assert np.array_equal(bits(yk), bits(ref)) and np.array_equal(bits(gk), bits(ref_b))


@pytest.mark.parametrize("xdt,rdt", [(BF16, F32), (BF16, BF16), (F32, F32), (F32, BF16)])
@pytest.mark.parametrize("shape", [(200, 4099), (33, 1023), (5, 13)])
def test_dropout_any_width_every_offset(xdt, rdt, shape):
    """Training at every offset, with elem_base chosen so that the body
    starts on a generator block (the pipeline) and so that it does not (the
    element-wise path); inference in place.  All bit-exact with the oracle."""
    rows, cols = shape
    x, b, r = W.dropout_inputs(rows, cols, xdt, rdt, seed=rows + cols)
    p, seed, offset = 0.3, 4321, 17
    ref_inf = O.bias_dropout_add_inference(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b))
    for k in offsets(xdt):
        head = (8 - k) % 8 if xdt == BF16 else (4 - k) % 4
        for elem_base in sorted({(8 - head) % 8, (8 - head) % 8 + 8 * 3 + 1, 5}):
            ref_out, ref_keep = O.bias_dropout_add_train(W.to_oracle(x), W.to_oracle(r), W.to_oracle(b), p=p,
                                                         seed=seed, offset=offset, elem_base=elem_base)
            out, keep = mfx.mfx_bias_dropout_add_train(
                at_offset(x, k), at_offset(b, k), at_offset(r, k), p, seed, offset, elem_base,
                out=empty_at(x.shape, xdt, k), keep_mask=empty_at(x.shape, torch.uint8, k))
            torch.cuda.synchronize()
            assert np.array_equal(keep.cpu().numpy(), ref_keep), (k, elem_base)
            assert np.array_equal(W.to_oracle(out), ref_out), (k, elem_base)
        xi = at_offset(x, k)
        mfx.mfx_bias_dropout_add_inference(xi, at_offset(b, (k + 1) % 8), at_offset(r, k))
        torch.cuda.synchronize()
        assert np.array_equal(W.to_oracle(xi), ref_inf), k
    assert mfx.mfx_device_error() == 0


def test_bias_gelu_bf16_odd_width_large_every_element():
    """A layer-sized odd width (4096 x 4099, bf16) through the pipeline at an
    offset of one element, every element against the oracle."""
    y, b, g = W.gelu_inputs(4096, 4099, BF16, seed=31)
    out = mfx.mfx_bias_gelu_fwd(at_offset(b, 1), at_offset(y, 1), out=empty_at(y.shape, BF16, 1))
    dy = mfx.mfx_bias_gelu_bwd(at_offset(g, 1), at_offset(b, 1), at_offset(y, 1), dy=empty_at(y.shape, BF16, 1))
    torch.cuda.synchronize()
    check(out, O.bias_gelu_fwd(W.to_oracle(y), W.to_oracle(b)), "fwd")
    ref, scale = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b), with_scale=True)
    check(dy, ref, "bwd", scale)


@pytest.mark.parametrize("rdt", [BF16, F32])
def test_dropout_misaligned_layer_shape_matches_aligned_bitwise(rdt):
    """The D2 layer shape, [4096 x 4] x 4096 bf16 x, p = 0.1: with every
    pointer one element off 16 bytes the body starts 7 elements in, off a
    generator block, so the kernel shares the blocks it draws across lanes,
    warps (through shared memory) and draws one more at each block's end.
    The whole output and mask equal the aligned call's, bit for bit."""
    x, b, r = W.dropout_inputs(16384, 4096, BF16, rdt, seed=21, device=DEV)
    out_a, keep_a = mfx.mfx_bias_dropout_add_train(x, b, r, 0.1, 1234, 5)
    out_m = empty_at(x.shape, BF16, 1)
    keep_m = empty_at(x.shape, torch.uint8, 1)
    mfx.mfx_bias_dropout_add_train(at_offset(x, 1), at_offset(b, 1), at_offset(r, 1), 0.1, 1234, 5,
                                   out=out_m, keep_mask=keep_m)
    torch.cuda.synchronize()
    assert torch.equal(keep_m, keep_a)
    assert torch.equal(out_m.view(torch.int16), out_a.view(torch.int16))
    assert mfx.mfx_device_error() == 0


def test_bias_gelu_layer_shape_pipeline_equals_elementwise_form_bitwise():
    """16384 x 16384 bf16 through the aligned pipeline and, with the
    pointers misaligned by different amounts, through the element-wise
    form (the same per-element arithmetic): forward and backward equal bit
    for bit over the whole tensor, so no unit of the persistent grid is
    dropped, repeated or given another column's bias."""
    y, b, g = W.gelu_inputs(16384, 16384, BF16, seed=41, device=DEV)
    out = mfx.mfx_bias_gelu_fwd(b, y)
    dy = mfx.mfx_bias_gelu_bwd(g, b, y)
    out_e = empty_at(y.shape, BF16, 2)
    dy_e = empty_at(y.shape, BF16, 3)
    mfx.mfx_bias_gelu_fwd(at_offset(b, 3), at_offset(y, 1), out=out_e)
    mfx.mfx_bias_gelu_bwd(at_offset(g, 5), at_offset(b, 0), at_offset(y, 1), dy=dy_e)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(dy.view(torch.int16), dy_e.view(torch.int16))
    assert mfx.mfx_device_error() == 0
