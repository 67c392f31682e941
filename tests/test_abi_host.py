"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/mfx.h declares, and rejects bad arguments before it
launches anything (every call below returns from host validation)."""
import ctypes as C
import os
import re

import pytest

import elementwise_epilogues_transformer_gb300 as mfx
from elementwise_epilogues_transformer_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mfx.h")

OK, NULL, SHAPE, DTYPE, PROB, ALIAS, CUDA = range(7)


@pytest.fixture(scope="module")
def L():
    B.build()
    return mfx.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mfx_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["mfx_bias_gelu_fwd", "mfx_bias_gelu_bwd", "mfx_bias_geglu_fwd", "mfx_bias_geglu_bwd",
              "mfx_bias_swiglu_fwd", "mfx_bias_swiglu_bwd", "mfx_bias_dropout_add_train",
              "mfx_bias_dropout_add_inference", "mfx_status_string", "mfx_last_cuda_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_binding_has_every_compute_entry_point():
    """The Python binding carries the C names: one function per compute
    entry point (the status, error and version queries are internal)."""
    internal = {"mfx_status_string", "mfx_last_cuda_error", "mfx_version"}
    for name in declared_functions():
        if name not in internal:
            assert callable(getattr(mfx, name, None)), name


def test_status_strings_and_version(L):
    for s in range(7):
        assert L.mfx_status_string(s)
    assert L.mfx_status_string(99) == b"unknown status"
    assert L.mfx_version() >> 16 == 1
    assert L.mfx_last_cuda_error() == 0


# Fake, never-dereferenced device addresses: every case below fails validation
# before any CUDA call.
A, B_, Cc, D = 0x10000, 0x20000000, 0x40000000, 0x60000000


def test_gelu_validation(L):
    f = L.mfx_bias_gelu_fwd
    assert f(7, 4, 8, None, A, B_, None) == DTYPE
    assert f(1, -1, 8, None, A, B_, None) == SHAPE
    assert f(1, 4, -8, None, A, B_, None) == SHAPE
    assert f(1, 2**62, 2**62, None, A, B_, None) == SHAPE
    assert f(1, 4, 8, None, None, B_, None) == NULL
    assert f(1, 4, 8, None, A, None, None) == NULL
    assert f(1, 0, 8, None, None, None, None) == OK        # empty: no-op
    assert f(1, 4, 0, None, None, None, None) == OK
    assert f(1, 4, 8, None, A, A + 2, None) == ALIAS        # partial overlap
    assert f(1, 4, 8, B_ + 8, A, B_, None) == ALIAS         # bias inside out
    g = L.mfx_bias_gelu_bwd
    assert g(1, 4, 8, None, None, A, B_, None) == NULL
    assert g(1, 4, 8, A, None, B_, A + 16, None) == ALIAS
    assert g(0, 4, 8, A, None, B_, B_ + 4, None) == ALIAS


def test_glu_validation(L):
    f = L.mfx_bias_swiglu_fwd
    assert f(3, 4, 8, A, None, None, B_, None) == DTYPE
    assert f(1, 4, -1, A, None, None, B_, None) == SHAPE
    assert f(1, 4, 8, None, None, None, B_, None) == NULL
    assert f(1, 4, 8, A, None, None, A + 8, None) == ALIAS  # out inside x
    assert f(1, 4, 8, A, None, B_ + 4, B_, None) == ALIAS   # weight inside out
    b = L.mfx_bias_swiglu_bwd
    assert b(1, 4, 8, A, B_, None, Cc, D, None, None) == NULL  # weight without dweight
    assert b(1, 4, 8, A, B_, None, None, B_ + 2, None, None) == ALIAS
    assert b(1, 4, 8, A, B_, None, Cc, D, D + 4, None) == ALIAS  # dweight inside dx
    gb = L.mfx_bias_geglu_bwd
    assert gb(1, 4, 8, None, B_, None, D, None) == NULL
    assert gb(1, 4, 8, D, B_, None, D, None) == ALIAS        # g inside dx
    assert L.mfx_bias_geglu_fwd(1, 0, 8, None, None, None, None) == OK


def test_dropout_validation(L):
    t = L.mfx_bias_dropout_add_train
    args = lambda **k: dict(dict(xd=1, rd=0, rows=4, cols=8, x=A, b=None, r=B_, p=0.1, seed=1,
                                  off=0, base=0, out=Cc, m=D, s=None), **k)
    call = lambda a: t(a["xd"], a["rd"], a["rows"], a["cols"], a["x"], a["b"], a["r"], a["p"],
                       a["seed"], a["off"], a["base"], a["out"], a["m"], a["s"])
    assert call(args(rd=5)) == DTYPE
    assert call(args(p=1.0)) == PROB
    assert call(args(p=-0.1)) == PROB
    assert call(args(p=float("nan"))) == PROB
    assert call(args(rows=-2)) == SHAPE
    assert call(args(base=2**64 - 4)) == SHAPE
    assert call(args(m=None)) == NULL
    assert call(args(r=None)) == NULL
    assert call(args(out=A + 2)) == ALIAS               # out partially over x
    assert call(args(out=B_)) == ALIAS                  # out over residual
    assert call(args(m=A + 4)) == ALIAS                 # mask over x
    assert call(args(m=Cc + 16)) == ALIAS               # mask over out
    assert call(args(rows=0, x=None, r=None, out=None, m=None)) == OK
    i = L.mfx_bias_dropout_add_inference
    assert i(1, 0, 4, 8, A, None, A + 8, 0.0, 0, 0, None) == ALIAS
    assert i(1, 0, 4, 8, A, A + 4, B_, 0.0, 0, 0, None) == ALIAS  # bias inside x
    assert i(1, 0, 4, 8, A, None, B_, 1.5, 0, 0, None) == PROB
    assert i(1, 0, 4, 8, None, None, B_, 0.0, 0, 0, None) == NULL


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(mfx, "_lib", None)
    monkeypatch.setattr(mfx, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mfx.lib()
