"""Seeded synthetic inputs and the workload shapes the library is measured on.

This module holds no arithmetic of the fused ops: it only draws random tensors
(normal or uniform, fp32, then cast) with fixed seeds and lists the shapes.
Both the GPU tests/benchmark and the CPU oracle consume what it draws.

Shapes follow the transformer layers the fused epilogues run in: the
bias-dropout-add residual of a [seq 4096 x batch 4 x hidden 4096] activation,
the bias-GeLU of a 16384-wide MLP, and the gated (GEGLU/SwiGLU) MLP input of
width 2 x 14336.  Values: activations and upstream gradients ~N(0, 1), biases
~N(0, 0.02), the per-token SwiGLU weight ~U(0, 1) in fp32.
"""
from dataclasses import dataclass, field

import torch

BIAS_STD = 0.02


def gen(seed: int, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, dtype, seed, std=1.0, device="cpu"):
    """N(0, std^2) drawn in fp32 from a seeded generator, then cast."""
    t = torch.randn(shape, generator=gen(seed, device), dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def uniform(shape, seed, device="cpu"):
    """U(0, 1) in fp32 from a seeded generator."""
    return torch.rand(shape, generator=gen(seed, device), dtype=torch.float32, device=device)


@dataclass(frozen=True)
class Workload:
    name: str
    op: str           # "gelu" | "glu" | "dropout" | "sqrelu" | "softmax"
    rows: int
    width: int        # cols for gelu/dropout, F (output width) for the GLU ops
    dtype: torch.dtype
    residual_dtype: torch.dtype = None
    p: float = 0.1
    seed: int = 0
    dropout_seed: int = 1234
    dropout_offset: int = 0
    note: str = field(default="", compare=False)


# The small fp32 case (the oracle runs it in seconds) and the three bf16
# layer-sized cases.
GELU_F32_SMALL = Workload("bias_gelu fp32 1024x4096", "gelu", 1024, 4096, torch.float32)
DROPOUT_BF16 = Workload("bias_dropout_add bf16 [4096x4]x4096, fp32 residual, p=0.1",
                        "dropout", 4096 * 4, 4096, torch.bfloat16,
                        residual_dtype=torch.float32, p=0.1)
GELU_BF16 = Workload("bias_gelu bf16 16384x16384", "gelu", 16384, 16384, torch.bfloat16)
GLU_BF16 = Workload("bias_swiglu/bias_geglu bf16 16384x(2x14336)", "glu", 16384, 14336,
                    torch.bfloat16)
# The weighted squared ReLU at the same MoE expert width (no gate half).
SQRELU_BF16 = Workload("weighted_squared_relu bf16 16384x14336", "sqrelu", 16384, 14336, torch.bfloat16)
# Attention-score softmax at the longest row the page's fused kernels take
# (sk = 4096): [b=2, np=32, sq=4096, sk=4096] with a padding mask, and the
# causal form on [attn_batches=64, 4096, 4096].  rows = b * np * sq.
SOFTMAX_BF16 = Workload("scaled_masked_softmax bf16 [2x32x4096x4096], pad mask [2x1x1x4096]", "softmax",
                        2 * 32 * 4096, 4096, torch.bfloat16)

SWEEP_TOKENS = (512, 4096, 32768, 65536)
SWEEP_HIDDEN = (1024, 4096, 4099, 8192, 16384)
SWEEP_P = (0.0, 0.1, 0.5)


def gelu_inputs(rows, cols, dtype, seed=0, device="cpu", with_bias=True):
    """y, bias, g for bias-GeLU forward/backward."""
    y = normal((rows, cols), dtype, seed, device=device)
    b = normal((cols,), dtype, seed + 1, std=BIAS_STD, device=device) if with_bias else None
    g = normal((rows, cols), dtype, seed + 2, device=device)
    return y, b, g


def glu_inputs(rows, F, dtype, seed=0, device="cpu", with_bias=True, with_weight=False):
    """x [rows, 2F], bias [2F], g [rows, F], weight [rows] fp32 for the GLU ops."""
    x = normal((rows, 2 * F), dtype, seed, device=device)
    b = normal((2 * F,), dtype, seed + 1, std=BIAS_STD, device=device) if with_bias else None
    g = normal((rows, F), dtype, seed + 2, device=device)
    w = uniform((rows,), seed + 3, device=device) if with_weight else None
    return x, b, g, w


def sqrelu_inputs(rows, cols, dtype, seed=0, device="cpu"):
    """x, g [rows, cols] (N(0, 1)) and the per-token router weight [rows]
    (U(0, 1) fp32) for the weighted squared ReLU."""
    x = normal((rows, cols), dtype, seed, device=device)
    g = normal((rows, cols), dtype, seed + 2, device=device)
    w = uniform((rows,), seed + 3, device=device)
    return x, g, w


def softmax_inputs(b, np_, sq, sk, dtype, seed=0, device="cpu", head_dim=128, mask=None):
    """Attention scores x [b, np, sq, sk] (q.k of unit-variance vectors of
    head_dim elements: N(0, head_dim)), the softmax scale 1/sqrt(head_dim),
    and an upstream gradient dy of x's shape (N(0, 1)).  mask: None, "pad"
    (additive [b, 1, 1, sk]: 0 on the first L_b keys, -inf after, L_b drawn
    uniformly from [sk/2, sk]) or "full" (additive [1, 1, sq, sk], N(0, 1)
    values)."""
    x = normal((b, np_, sq, sk), dtype, seed, std=float(head_dim) ** 0.5, device=device)
    dy = normal((b, np_, sq, sk), dtype, seed + 1, device=device)
    m = None
    if mask == "pad":
        g = gen(seed + 2)
        lengths = torch.randint(max(1, sk // 2), sk + 1, (b,), generator=g)
        keep = torch.arange(sk)[None, :] < lengths[:, None]
        m = torch.where(keep, 0.0, float("-inf")).to(dtype).reshape(b, 1, 1, sk).to(device)
    elif mask == "full":
        m = normal((1, 1, sq, sk), dtype, seed + 3, device=device)
    return x, m, dy, 1.0 / float(head_dim) ** 0.5


def dropout_inputs(rows, cols, dtype, residual_dtype, seed=0, device="cpu", with_bias=True):
    """x, bias (x's dtype), residual (its own dtype) for bias-dropout-add."""
    x = normal((rows, cols), dtype, seed, device=device)
    b = normal((cols,), dtype, seed + 1, std=BIAS_STD, device=device) if with_bias else None
    r = normal((rows, cols), residual_dtype, seed + 2, device=device)
    return x, b, r


def to_oracle(t):
    """A torch tensor as the oracle's numpy array (bf16 as raw uint16 bits)."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16").copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    raise TypeError(f"unsupported dtype {t.dtype}")
