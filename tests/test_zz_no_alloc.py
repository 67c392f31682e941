"""The allocation-free bias-GeLU backward with bias gradient
(mfx_bias_gelu_bwd_dbias_noalloc), called through the C ABI.

It is for callers that cannot hand the library a workspace: code whose device
memory all belongs to a pool that gives library calls no scratch, code where
a device allocation (which may synchronise the device) is not acceptable, and
C callers without a device allocator.  The library keeps one fixed scratch
array per device instead, so its results must equal those of the workspace
entry point bit for bit whenever both use the same partial layout.  Calls in
a row share that array: the first call here leaves nonzero partials in more
of it than the next ones need, so a slot a later call read without writing
would change its bits.  This file is collected last so that a run stopping
at the first failure has run everything else."""
import ctypes as C

import numpy as np
import pytest
import torch

import dbias_order as DBO
import elementwise_epilogues_transformer_gb300 as mfx
import oracle as O
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bf16_ulp, bits, f32_ulp, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 4 << 20          # the array's documented size


@pytest.fixture(scope="module")
def L():
    B.build()
    return mfx.lib()


def call_noalloc(L, g, b, y):
    rows, cols = y.shape
    dy = torch.empty_like(y)
    db = torch.empty(cols, dtype=y.dtype, device=DEV)
    st = L.mfx_bias_gelu_bwd_dbias_noalloc(mfx.dtype_code(y.dtype), rows, cols, g.data_ptr(), b.data_ptr(),
                                           y.data_ptr(), dy.data_ptr(), db.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == 0, mfx.STATUS.get(st, st)
    return dy, db


def workspace_call(g, b, y):
    """The workspace entry point with a NaN-filled workspace; returns dy,
    dbias and the partial count J it wrote."""
    box = {}

    def alloc(n):
        box["ws"] = DBO.nan_workspace(n, DEV)
        return box["ws"]

    dy, db = mfx.mfx_bias_gelu_bwd_dbias(g, b, y, workspace=alloc)
    torch.cuda.synchronize()
    return dy, db, DBO.partials_written(box["ws"], y.shape[1])


def test_noalloc_equals_workspace_entry_point_over_calls_in_a_row(L):
    # (rows, cols, dtype, seed): the first writes the most partial slots
    # (about 2.5 MB of the array), the later ones fewer, over its stale values
    cases = [(8192, 1024, torch.bfloat16, 1), (4096, 4096, torch.bfloat16, 2),
             (300, 1000, torch.float32, 3), (200, 4096, torch.bfloat16, 4)]
    slots = []
    for rows, cols, dtype, seed in cases:
        y, b, g = W.gelu_inputs(rows, cols, dtype, seed=seed, device=DEV)
        dy_ref, db_ref, J = workspace_call(g, b, y)
        slots.append(J * cols)
        dy, db = call_noalloc(L, g, b, y)
        torch.cuda.synchronize()
        assert np.array_equal(bits(dy), bits(dy_ref)), (rows, cols)
        assert np.array_equal(bits(db), bits(db_ref)), (rows, cols)
    assert slots[0] == max(slots) and slots[0] * 4 <= SCRATCH_BYTES
    assert mfx.mfx_device_error() == 0


def test_noalloc_against_oracle_column_sums(L):
    """dbias against the oracle: the column sums of the oracle's own gradient,
    within the summation order's bound plus each stored element's tolerance."""
    rows, cols = 300, 1000
    for dtype in (torch.float32, torch.bfloat16):
        y, b, g = W.gelu_inputs(rows, cols, dtype, seed=5)
        yd, bd, gd = y.to(DEV), b.to(DEV), g.to(DEV)
        _, _, J = workspace_call(gd, bd, yd)
        dy, db = call_noalloc(L, gd, bd, yd)
        torch.cuda.synchronize()
        ref = O.bias_gelu_bwd(W.to_oracle(g), W.to_oracle(y), W.to_oracle(b))
        name = "bf16" if dtype == torch.bfloat16 else "f32"
        rs, mag = O.column_sums(ref, name)
        got = to_f64(db)
        elem = bf16_ulp(ref) if name == "bf16" else np.maximum(1e-6, 2 * f32_ulp(ref))
        tol = DBO.tolerance(got, rs, mag, rows, J, name == "bf16") + elem.sum(axis=0)
        assert np.all(np.abs(got - rs) <= tol), float(np.max(np.abs(got - rs) / tol))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(33, 4104), (63, 16392), (5, 65544)])
def test_noalloc_wide_rows(L, dtype, shape):
    """Wide rows: where the workspace entry point's partials fit the array,
    both calls give the same bits; where they do not (a device with more
    resident threads per SM than this one), the call takes the
    row-interleaved layout, min(rows, 64) partials per column: dy is still
    the same bits, and dbias is that layout's documented order (bit for bit)
    and within the bound of the exact sum."""
    rows, cols = shape
    y, b, g = W.gelu_inputs(rows, cols, dtype, seed=6, device=DEV)
    dy_ref, db_ref, J_ws = workspace_call(g, b, y)
    dy, db = call_noalloc(L, g, b, y)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dy), bits(dy_ref))
    if J_ws * cols * 4 <= SCRATCH_BYTES:
        assert np.array_equal(bits(db), bits(db_ref))
        return
    st32 = dy.float().cpu().numpy()
    J = min(rows, 64)
    rep = torch.from_numpy(DBO.replay(st32, J)).to(dtype)
    assert np.array_equal(bits(rep), bits(db))
    exact, mag = DBO.column_sums(st32)
    got = to_f64(db)
    assert np.all(np.abs(got - exact) <= DBO.tolerance(got, exact, mag, rows, J, dtype == torch.bfloat16))


def test_noalloc_python_binding(L):
    y, b, g = W.gelu_inputs(512, 2048, torch.bfloat16, seed=3, device=DEV)
    dy_ref, db_ref = mfx.mfx_bias_gelu_bwd_dbias(g, b, y)
    dy, db = mfx.mfx_bias_gelu_bwd_dbias_noalloc(g, b, y)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dy), bits(dy_ref)) and np.array_equal(bits(db), bits(db_ref))


def test_noalloc_rejects_problems_beyond_its_scratch(L):
    cols = 1 << 20                               # 64 lanes x 2^20 columns x 4 B > 4 MiB
    y = torch.zeros(64, cols, dtype=torch.bfloat16, device=DEV)
    db = torch.empty(cols, dtype=torch.bfloat16, device=DEV)
    st = L.mfx_bias_gelu_bwd_dbias_noalloc(1, 64, cols, y.data_ptr(), None, y.data_ptr(), y.data_ptr(),
                                           db.data_ptr(), None)
    assert st == 8
