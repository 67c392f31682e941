"""The allocation-free bias-GeLU backward with bias gradient
(mfx_bias_gelu_bwd_dbias_noalloc), called through the C ABI: it serves
callers that cannot give the library a workspace (the library keeps a fixed
scratch array instead), so its results must equal those of the workspace
entry point.  Two calls in a row check that the shared array left over from
one call does not leak into the next.  This file is collected last so that
a run stopping at the first failure has run everything else."""
import ctypes as C

import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W
from parity import bf16_ulp, f32_ulp, to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


def close(a, b, dtype):
    """Within the tolerance the parity tests use for the two outputs."""
    av, bv = to_f64(a), to_f64(b)
    ulp = bf16_ulp if dtype == torch.bfloat16 else f32_ulp
    return np.all(np.abs(av - bv) <= ulp(bv))


def test_noalloc_matches_workspace_entry_point_two_calls(L):
    cases = [(4096, 4096, torch.bfloat16, 1), (300, 1000, torch.float32, 2)]
    for rows, cols, dtype, seed in cases:        # two calls in a row, different shapes
        y, b, g = W.gelu_inputs(rows, cols, dtype, seed=seed, device=DEV)
        dy_ref, db_ref = mfx.mfx_bias_gelu_bwd_dbias(g, b, y)
        dy, db = call_noalloc(L, g, b, y)
        torch.cuda.synchronize()
        assert close(dy, dy_ref, dtype)
        assert close(db, db_ref, dtype)
    assert mfx.mfx_device_error() == 0


def test_noalloc_python_binding(L):
    y, b, g = W.gelu_inputs(512, 2048, torch.bfloat16, seed=3, device=DEV)
    dy_ref, db_ref = mfx.mfx_bias_gelu_bwd_dbias(g, b, y)
    dy, db = mfx.mfx_bias_gelu_bwd_dbias_noalloc(g, b, y)
    torch.cuda.synchronize()
    assert close(dy, dy_ref, torch.bfloat16) and close(db, db_ref, torch.bfloat16)


def test_noalloc_rejects_problems_beyond_its_scratch(L):
    cols = 1 << 20                               # 64 lanes x 2^20 columns x 4 B > 4 MiB
    y = torch.zeros(64, cols, dtype=torch.bfloat16, device=DEV)
    db = torch.empty(cols, dtype=torch.bfloat16, device=DEV)
    st = L.mfx_bias_gelu_bwd_dbias_noalloc(1, 64, cols, y.data_ptr(), None, y.data_ptr(), y.data_ptr(),
                                           db.data_ptr(), None)
    assert st == 8
