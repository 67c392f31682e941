"""Every kind of launch the library makes can be captured in a CUDA graph and
replayed: the bulk-copy pipelines, the row pipelines of the softmax (whose
launcher sets the kernel's shared-memory attribute), the fused bias
gradients (whose finish kernel is a programmatic dependent launch) and the
generic fallbacks.  Replays give the eager call's bits."""
import numpy as np
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
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


def _ops():
    """(name, fn) pairs writing into preallocated outputs; fn() runs one call."""
    y, b, g = (t.to(DEV) for t in W.gelu_inputs(96, 4096, BF16, seed=1))
    yu, bu, gu = (t.to(DEV) for t in W.gelu_inputs(7, 4099, BF16, seed=2))     # generic path
    x, b2, g2, w = (t.to(DEV) for t in W.glu_inputs(64, 1024, BF16, seed=3, with_weight=True))
    xd, bd, rd = (t.to(DEV) for t in W.dropout_inputs(64, 4096, BF16, F32, seed=4))
    xs, _, dys, scale = W.softmax_inputs(1, 3, 512, 512, BF16, seed=5)
    xs, dys = xs[0].to(DEV), dys[0].to(DEV)
    o = {
        "gelu": torch.empty_like(y), "dy": torch.empty_like(y), "db": torch.empty(4096, dtype=BF16, device=DEV),
        "gelu_u": torch.empty_like(yu), "glu": torch.empty(64, 1024, dtype=BF16, device=DEV),
        "dx": torch.empty_like(x), "dw": torch.empty(64, dtype=F32, device=DEV),
        "od": torch.empty_like(xd), "keep": torch.empty(xd.shape, dtype=torch.uint8, device=DEV),
        "ys": torch.empty_like(xs), "dxs": torch.empty_like(xs),
        "dxd": torch.empty_like(xd), "dres": torch.empty(xd.shape, dtype=F32, device=DEV),
        "dbd": torch.empty(4096, dtype=BF16, device=DEV),
    }
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=DEV)
    ops = [
        ("gelu_fwd", lambda: mfx.mfx_bias_gelu_fwd(b, y, out=o["gelu"])),
        ("gelu_bwd_dbias", lambda: mfx.mfx_bias_gelu_bwd_dbias(g, b, y, dy=o["dy"], dbias=o["db"], workspace=ws)),
        ("gelu_fwd_generic", lambda: mfx.mfx_bias_gelu_fwd(bu, yu, out=o["gelu_u"])),
        ("swiglu_w_fwd", lambda: mfx.mfx_bias_swiglu_fwd(x, b2, w, out=o["glu"])),
        ("swiglu_w_bwd", lambda: mfx.mfx_bias_swiglu_bwd(g2, x, b2, w, dx=o["dx"], dweight=o["dw"])),
        ("dropout_train", lambda: mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.1, 1234, 0, out=o["od"],
                                                               keep_mask=o["keep"])),
        ("dropout_bwd_dbias", lambda: mfx.mfx_bias_dropout_add_bwd_dbias(
            o["od"], None, 0.1, 1234, 0, dx=o["dxd"], dresidual=o["dres"], dbias=o["dbd"], workspace=ws)),
        ("softmax_causal_fwd", lambda: mfx.mfx_scaled_upper_triang_masked_softmax_fwd(xs, scale, y=o["ys"])),
        ("softmax_causal_bwd", lambda: mfx.mfx_scaled_upper_triang_masked_softmax_bwd(dys, o["ys"], scale,
                                                                                      dx=o["dxs"])),
    ]
    return ops, o


def test_graph_replay_matches_eager():
    ops, o = _ops()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _, fn in ops:      # eager, on the side stream (also warms up every launcher)
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in o.items()}
    for v in o.values():
        v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _, fn in ops:
            fn()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for k, v in o.items():
        assert np.array_equal(bits(v), bits(eager[k])), k
    assert mfx.mfx_device_error() == 0


# A step of forward and backward calls at layer-like widths, including the
# forms added for odd widths (the GLU realigning ring, F = 4099), the
# byte-mask dropout backward's bulk stores and the masked softmax.
def workspace_for(fn):
    """A workspace of the size the call asks for (queried outside the graph)."""
    box = {}

    def alloc(n):
        box["ws"] = torch.empty(n, dtype=torch.uint8, device=DEV)
        return box["ws"]

    fn(alloc)
    return box["ws"]


def make_step(T, H, F):
    y, b, g = W.gelu_inputs(T, H, BF16, seed=1, device=DEV)
    x, bg, gg, w = W.glu_inputs(T, F, BF16, seed=2, device=DEV, with_weight=True)
    xd, bd, rd = W.dropout_inputs(T, H, BF16, torch.float32, seed=3, device=DEV)
    gd = W.normal((T, H), BF16, 4, device=DEV)
    sx, smask, sdy, scale = W.softmax_inputs(2, 4, 64, 128, BF16, seed=5, device=DEV, mask="pad")
    o = {
        "gelu": torch.empty_like(y), "gelu_dy": torch.empty_like(y), "gelu_db": torch.empty(H, dtype=BF16, device=DEV),
        "geglu": torch.empty(T, F, dtype=BF16, device=DEV), "geglu_dx": torch.empty_like(x),
        "swiglu_w": torch.empty(T, F, dtype=BF16, device=DEV), "swiglu_dx": torch.empty_like(x),
        "swiglu_dw": torch.empty(T, dtype=torch.float32, device=DEV),
        "bda": torch.empty_like(xd), "keep": torch.empty(T, H, dtype=torch.uint8, device=DEV),
        "bda_dx": torch.empty_like(xd), "bda_dres": torch.empty(T, H, dtype=torch.float32, device=DEV),
        "sm": torch.empty_like(sx), "sm_dx": torch.empty_like(sx),
    }
    ws = workspace_for(lambda a: mfx.mfx_bias_gelu_bwd_dbias(g, b, y, dy=o["gelu_dy"], dbias=o["gelu_db"],
                                                            workspace=a))

    def step():
        mfx.mfx_bias_gelu_fwd(b, y, out=o["gelu"])
        mfx.mfx_bias_gelu_bwd_dbias(g, b, y, dy=o["gelu_dy"], dbias=o["gelu_db"], workspace=ws)
        mfx.mfx_bias_geglu_fwd(x, bg, out=o["geglu"])
        mfx.mfx_bias_geglu_bwd(gg, x, bg, dx=o["geglu_dx"])
        mfx.mfx_bias_swiglu_fwd(x, bg, w, out=o["swiglu_w"])
        mfx.mfx_bias_swiglu_bwd(gg, x, bg, w, dx=o["swiglu_dx"], dweight=o["swiglu_dw"])
        mfx.mfx_bias_dropout_add_train(xd, bd, rd, 0.1, 1234, 7, out=o["bda"], keep_mask=o["keep"])
        mfx.mfx_bias_dropout_add_bwd(gd, o["keep"], 0.1, dx=o["bda_dx"], dresidual=o["bda_dres"])
        mfx.mfx_scaled_masked_softmax_fwd(sx, scale, smask, y=o["sm"])
        mfx.mfx_scaled_masked_softmax_bwd(sdy, o["sm"], scale, dx=o["sm_dx"])

    return step, o


@pytest.mark.parametrize("T,H,F", [(64, 1024, 1024), (512, 4096, 4099)])
def test_layer_step_in_a_graph_matches_eager(T, H, F):
    step, o = make_step(T, H, F)
    step()                                   # eager (also fills the host-side launch plans)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in o.items()}
    for v in o.values():
        v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for k, v in o.items():
        assert torch.equal(v.view(torch.uint8), eager[k].view(torch.uint8)), k
    assert mfx.mfx_device_error() == 0
