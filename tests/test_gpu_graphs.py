"""The entry points inside a CUDA graph.

A caller whose steps are small (decode-sized tensors) is bound by the launch
rate, and the usual answer is to capture the step once into a CUDA graph and
replay it.  The library's calls take the caller's stream, allocate nothing
when their outputs (and, for the fused bias gradients, the workspace) are
given, and keep their launch plans on the host, so they can be captured:
this file captures a step of forward and backward calls (dropout with its
mask, the fused bias gradients with a caller's workspace, softmax), replays
it, and requires every output to equal the eager call's bit for bit.  The
allocation-free entry point is not part of it."""
import pytest
import torch

import elementwise_epilogues_transformer_gb300 as mfx
from elementwise_epilogues_transformer_gb300 import build as B
from elementwise_epilogues_transformer_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()
    mfx.lib()


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
def test_step_in_a_cuda_graph_matches_eager(T, H, F):
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
