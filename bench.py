#!/usr/bin/env python3
"""Benchmark of the fused transformer MLP / residual epilogues (libmfx).

One step runs every fused op once, in bf16, on layer-sized synthetic inputs:
  bias-GeLU forward and backward          y [16384 x 16384]
  bias-GEGLU forward and backward         x [16384 x 2*14336]
  bias-SwiGLU forward and backward        x [16384 x 2*14336], plain and with
                                          the per-token fp32 weight [16384]
  bias-dropout-add train and inference    x [4096*4 x 4096], fp32 residual,
                                          p = 0.1, Philox seed 1234, offset 0
`value` is the whole step's achieved HBM bandwidth: the algorithmic bytes of
all ops (one read of every input, one write of every output) divided by the
device time of the step, summed over ranks (each rank processes its own
batch: weak scaling).  Every input is larger than L2 (129 MB), so nothing is
served from L2 between iterations.

--impl reference times the CPU oracle (oracle/) on bounded row samples of
the same workload; the default run also reports that oracle as cpu_baseline.
"""
import argparse
import dataclasses
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "achieved HBM GB/s and % of GB300 peak per fused op (bf16 fwd+bwd); elements/s"
WORKLOAD = ("fused MLP+residual epilogue step, bf16: bias_gelu fwd+bwd 16384x16384; "
            "bias_geglu, bias_swiglu and weighted bias_swiglu fwd+bwd 16384x(2x14336); "
            "bias_dropout_add train+inference [4096x4]x4096 fp32 residual p=0.1")
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mfx", "reference"], default="mfx")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="copy streams per direction in the end-to-end run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target oracle CPU time for the cpu_baseline sample")
    ap.add_argument("--only", default="", help="comma-separated op names (profiling runs)")
    ap.add_argument("--next-only", default="",
                    help="comma-separated names of the ops beyond the step to time (profiling runs)")
    ap.add_argument("--rows-scale", type=float, default=1.0,
                    help="scale every workload's row count (profiling captures on smaller cases; "
                         "not a headline configuration)")
    ap.add_argument("--no-isolated", action="store_true",
                    help="skip timing each step op alone, back to back (per_op_isolated: each launch then "
                         "pays only its own predecessor's L2 write-back, where inside the step it pays "
                         "the previous op's)")
    ap.add_argument("--no-next", action="store_true",
                    help="skip timing the ops beyond the step (next_per_op)")
    ap.add_argument("--largest", action="store_true",
                    help="also time each step op alone at the sweep's largest row, 65536 x 16384 "
                         "(largest_per_op)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the shape sweep (tokens x hidden, both dtypes, every op; medians of 20)")
    ap.add_argument("--sweep-reps", type=int, default=20, help="timed launches per sweep entry (median)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU under torchrun; replicas of the
# per-GPU workload, each on its own shard of a global batch)
# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the step: every op, its algorithmic bytes and its inputs/outputs
# ---------------------------------------------------------------------------
class Op:
    def __init__(self, name, kernel, fn, nbytes, elems, inputs, outputs, oracle=None):
        self.name, self.kernel, self.fn = name, kernel, fn
        self.nbytes, self.elems = nbytes, elems
        self.inputs, self.outputs = inputs, outputs   # tensors copied in/out by the e2e run
        self.oracle = oracle                          # callable(rows) -> (bytes, seconds)


ROWS_SCALE = 1.0  # set from --rows-scale


def scaled(w):
    """The workload with its row count scaled by --rows-scale."""
    if ROWS_SCALE == 1.0:
        return w
    return dataclasses.replace(w, rows=max(8, int(w.rows * ROWS_SCALE)))


# The largest row of the shape sweep (tokens x hidden; the GLU width F is
# the hidden size, so its input is 2 x 16384 wide).
LARGEST = {"rows": 65536, "width": 16384}


def build_step(dev, rank, only=(), largest=False):
    import elementwise_epilogues_transformer_gb300 as mfx
    from elementwise_epilogues_transformer_gb300 import workloads as W
    from elementwise_epilogues_transformer_gb300.sharding import shard_elem_base

    bf = torch.bfloat16
    seed = 1000 * rank
    ops = []

    def want(name):
        return not only or name in only

    # bias-GeLU
    big = (lambda w: dataclasses.replace(w, **LARGEST)) if largest else scaled
    wg = big(W.GELU_BF16)
    if want("bias_gelu_fwd") or want("bias_gelu_bwd"):
        y, b, g = W.gelu_inputs(wg.rows, wg.width, bf, seed=seed, device=dev)
        out, dy = torch.empty_like(y), torch.empty_like(y)
        n = wg.rows * wg.width
        if want("bias_gelu_fwd"):
            ops.append(Op("bias_gelu_fwd", "gelu_pipe<bf16,fwd>",
                          lambda: mfx.mfx_bias_gelu_fwd(b, y, out=out), 4 * n + 2 * wg.width, n,
                          [y, b], [out], oracle=("gelu_fwd", (y, b, g))))
        if want("bias_gelu_bwd"):
            ops.append(Op("bias_gelu_bwd", "gelu_pipe<bf16,bwd>",
                          lambda: mfx.mfx_bias_gelu_bwd(g, b, y, dy=dy), 6 * n + 2 * wg.width, n,
                          [g, y, b], [dy], oracle=("gelu_bwd", (y, b, g))))

    # GLU family
    wl = big(W.GLU_BF16)
    names = ["bias_geglu_fwd", "bias_geglu_bwd", "bias_swiglu_fwd", "bias_swiglu_bwd",
             "bias_swiglu_w_fwd", "bias_swiglu_w_bwd"]
    if any(want(nm) for nm in names):
        x, b2, g2, w = W.glu_inputs(wl.rows, wl.width, bf, seed=seed + 10, device=dev, with_weight=True)
        # every op has its own output buffers, so that the end-to-end run can
        # copy one op's result back while the next op computes
        o2g, o2s, o2w = (torch.empty(wl.rows, wl.width, dtype=bf, device=dev) for _ in range(3))
        dxg, dxs, dxw = (torch.empty_like(x) for _ in range(3))
        dw = torch.empty(wl.rows, dtype=torch.float32, device=dev)
        m = wl.rows * wl.width
        fb, bb = 6 * m + 4 * wl.width, 10 * m + 4 * wl.width
        table = [
            ("bias_geglu_fwd", "glu_pipe<bf16,GEGLU,fwd>", lambda: mfx.mfx_bias_geglu_fwd(x, b2, out=o2g),
             fb, [x, b2], [o2g], ("geglu_fwd", (x, b2, g2, None))),
            ("bias_geglu_bwd", "glu_pipe<bf16,GEGLU,bwd>", lambda: mfx.mfx_bias_geglu_bwd(g2, x, b2, dx=dxg),
             bb, [g2, x, b2], [dxg], ("geglu_bwd", (x, b2, g2, None))),
            ("bias_swiglu_fwd", "glu_pipe<bf16,SWIGLU,fwd>", lambda: mfx.mfx_bias_swiglu_fwd(x, b2, out=o2s),
             fb, [x, b2], [o2s], ("swiglu_fwd", (x, b2, g2, None))),
            ("bias_swiglu_bwd", "glu_pipe<bf16,SWIGLU,bwd>",
             lambda: mfx.mfx_bias_swiglu_bwd(g2, x, b2, dx=dxs), bb, [g2, x, b2], [dxs],
             ("swiglu_bwd", (x, b2, g2, None))),
            ("bias_swiglu_w_fwd", "glu_pipe<bf16,SWIGLU,weighted,fwd>",
             lambda: mfx.mfx_bias_swiglu_fwd(x, b2, w, out=o2w), fb + 4 * wl.rows, [x, b2, w], [o2w],
             ("swiglu_fwd", (x, b2, g2, w))),
            ("bias_swiglu_w_bwd", "swiglu_bwd_weighted_pipe<bf16>",
             lambda: mfx.mfx_bias_swiglu_bwd(g2, x, b2, w, dx=dxw, dweight=dw), bb + 8 * wl.rows,
             [g2, x, b2, w], [dxw, dw], ("swiglu_bwd", (x, b2, g2, w))),
        ]
        for name, kern, fn, nb, ins, outs, orc in table:
            if want(name):
                ops.append(Op(name, kern, fn, nb, m, ins, outs, oracle=orc))

    # bias-dropout-add
    wd = big(W.DROPOUT_BF16)
    if want("bias_dropout_add_train") or want("bias_dropout_add_inference"):
        xd, bd, rd = W.dropout_inputs(wd.rows, wd.width, bf, wd.residual_dtype, seed=seed + 20, device=dev)
        xi = xd.clone()
        od = torch.empty_like(xd)
        keep = torch.empty(xd.shape, dtype=torch.uint8, device=dev)
        n = wd.rows * wd.width
        # this rank's rows are rows [rank*R, (rank+1)*R) of the global batch
        base = shard_elem_base(rank * wd.rows, wd.width)
        if want("bias_dropout_add_train"):
            ops.append(Op("bias_dropout_add_train", "bda_pipe<bf16,f32,train>",
                          lambda: mfx.mfx_bias_dropout_add_train(xd, bd, rd, wd.p, wd.dropout_seed,
                                                                 wd.dropout_offset, base, out=od,
                                                                 keep_mask=keep),
                          9 * n + 2 * wd.width, n, [xd, bd, rd], [od, keep],
                          oracle=("bda_train", (xd, bd, rd, base))))
        if want("bias_dropout_add_inference"):
            ops.append(Op("bias_dropout_add_inference", "bda_pipe<bf16,f32,inference>",
                          lambda: mfx.mfx_bias_dropout_add_inference(xi, bd, rd, wd.p, wd.dropout_seed,
                                                                     wd.dropout_offset),
                          8 * n + 2 * wd.width, n, [xi, bd, rd], [xi],
                          oracle=("bda_inference", (xi, bd, rd, base))))
    return ops


def build_next(dev, only=()):
    """Ops beyond the step (backward of bias-dropout-add, fused bias
    gradients, the weighted squared ReLU, scale-mask-softmax), timed
    separately; same byte accounting (algorithmic bytes: every input element
    the op must read, every output element it writes)."""
    import elementwise_epilogues_transformer_gb300 as mfx
    from elementwise_epilogues_transformer_gb300 import workloads as W

    bf = torch.bfloat16
    ops = []
    wd = scaled(W.DROPOUT_BF16)
    n = wd.rows * wd.width
    g = W.normal((wd.rows, wd.width), bf, 31, device=dev)
    x, b, r = W.dropout_inputs(wd.rows, wd.width, bf, wd.residual_dtype, seed=30, device=dev)
    _, keep = mfx.mfx_bias_dropout_add_train(x, b, r, wd.p, wd.dropout_seed, wd.dropout_offset)
    dx = torch.empty_like(g)
    dres = torch.empty(g.shape, dtype=torch.float32, device=dev)
    dbd = torch.empty(wd.width, dtype=bf, device=dev)
    ops.append(Op("bias_dropout_add_bwd(mask)", "bda_bwd_pipe<bf16,f32,mask>",
                  lambda: mfx.mfx_bias_dropout_add_bwd(g, keep, wd.p, dx=dx, dresidual=dres),
                  (2 + 1 + 2 + 4) * n, n, [], []))
    ops.append(Op("bias_dropout_add_bwd(regen)", "bda_bwd_pipe<bf16,f32,regen>",
                  lambda: mfx.mfx_bias_dropout_add_bwd(g, None, wd.p, wd.dropout_seed, wd.dropout_offset,
                                                       dx=dx, dresidual=dres),
                  (2 + 2 + 4) * n, n, [], []))
    od = torch.empty_like(x)
    kbits = torch.empty((n + 7) // 8, dtype=torch.uint8, device=dev)
    ops.append(Op("bias_dropout_add_train(packed mask)", "bda_pipe<bf16,f32,train,packed>",
                  lambda x=x, b=b, r=r: mfx.mfx_bias_dropout_add_train_packed(
                      x, b, r, wd.p, wd.dropout_seed, wd.dropout_offset, out=od, keep_bits=kbits),
                  (2 + 4 + 2) * n + (n + 7) // 8 + 2 * wd.width, n, [], []))
    ops.append(Op("bias_dropout_add_train(byte mask)", "bda_pipe<bf16,f32,train>",
                  lambda x=x, b=b, r=r: mfx.mfx_bias_dropout_add_train(
                      x, b, r, wd.p, wd.dropout_seed, wd.dropout_offset, out=od, keep_mask=keep),
                  (2 + 4 + 2 + 1) * n + 2 * wd.width, n, [], []))
    ops.append(Op("bias_dropout_add_bwd(packed mask)", "bda_bwd_pipe<bf16,f32,packed>",
                  lambda: mfx.mfx_bias_dropout_add_bwd_packed(g, kbits, wd.p, dx=dx, dresidual=dres),
                  (2 + 2 + 4) * n + (n + 7) // 8, n, [], []))
    wsd = torch.empty(16 << 20, dtype=torch.uint8, device=dev)
    ops.append(Op("bias_dropout_add_bwd_dbias(regen)", "bda_bwd_pipe<bf16,f32,regen,dbias>",
                  lambda: mfx.mfx_bias_dropout_add_bwd_dbias(g, None, wd.p, wd.dropout_seed, wd.dropout_offset,
                                                             dx=dx, dresidual=dres, dbias=dbd, workspace=wsd),
                  (2 + 2 + 4) * n + 2 * wd.width, n, [], []))
    wg = scaled(W.GELU_BF16)
    m = wg.rows * wg.width
    y, bg, gg = W.gelu_inputs(wg.rows, wg.width, bf, seed=40, device=dev)
    dy = torch.empty_like(y)
    dbg = torch.empty(wg.width, dtype=bf, device=dev)
    ops.append(Op("bias_gelu_bwd_dbias", "gelu_pipe<bf16,bwd,dbias>",
                  lambda: mfx.mfx_bias_gelu_bwd_dbias(gg, bg, y, dy=dy, dbias=dbg, workspace=wsd),
                  6 * m + 4 * wg.width, m, [], []))
    wl = scaled(W.GLU_BF16)
    q = wl.rows * wl.width
    xg, b2, g2, _ = W.glu_inputs(wl.rows, wl.width, bf, seed=50, device=dev)
    dx2 = torch.empty_like(xg)
    db2 = torch.empty(2 * wl.width, dtype=bf, device=dev)
    ops.append(Op("bias_geglu_bwd_dbias", "glu_pipe<bf16,GEGLU,bwd,dbias>",
                  lambda: mfx.mfx_bias_geglu_bwd_dbias(g2, xg, b2, dx=dx2, dbias=db2, workspace=wsd),
                  10 * q + 8 * wl.width, q, [], []))
    ws_ = scaled(W.SQRELU_BF16)
    k = ws_.rows * ws_.width
    xs, gs, w_s = W.sqrelu_inputs(ws_.rows, ws_.width, bf, seed=60, device=dev)
    fs = torch.empty_like(xs)
    dxs = torch.empty_like(xs)
    dws = torch.empty(ws_.rows, dtype=torch.float32, device=dev)
    ops.append(Op("weighted_squared_relu_fwd", "sqrelu_fwd_pipe<bf16>",
                  lambda: mfx.mfx_weighted_squared_relu_fwd(xs, w_s, out=fs),
                  4 * k + 4 * ws_.rows, k, [], []))
    ops.append(Op("weighted_squared_relu_bwd", "sqrelu_bwd_pipe<bf16>",
                  lambda: mfx.mfx_weighted_squared_relu_bwd(gs, xs, w_s, dx=dxs, dweight=dws),
                  6 * k + 8 * ws_.rows, k, [], []))
    # scale-mask-softmax: padding-masked and causal, forward and backward
    sm = W.SOFTMAX_BF16
    b, heads, sq, sk = 2, max(1, int(32 * ROWS_SCALE)), 4096, sm.width
    N = b * heads * sq * sk
    xq, mq, dyq, scale = W.softmax_inputs(b, heads, sq, sk, bf, seed=70, device=dev, mask="pad")
    yq = torch.empty_like(xq)
    dxq = torch.empty_like(xq)
    ops.append(Op("scaled_masked_softmax_fwd(pad)", "softmax_fwd_rowpipe<bf16,mask>",
                  lambda: mfx.mfx_scaled_masked_softmax_fwd(xq, scale, mq, y=yq),
                  4 * N + 2 * b * sk, N, [], []))
    ops.append(Op("scaled_masked_softmax_bwd", "softmax_bwd_rowpipe<bf16>",
                  lambda: mfx.mfx_scaled_masked_softmax_bwd(dyq, yq, scale, dx=dxq),
                  6 * N, N, [], []))
    xc, yc, dyc, dxc = (t.view(b * heads, sq, sk) for t in (xq, yq, dyq, dxq))
    valid = b * heads * sq * (sq + 1) // 2
    ops.append(Op("scaled_upper_triang_masked_softmax_fwd", "softmax_fwd_rowpipe<bf16,causal>",
                  lambda: mfx.mfx_scaled_upper_triang_masked_softmax_fwd(xc, scale, y=yc),
                  2 * valid + 2 * N, N, [], []))
    ops.append(Op("scaled_upper_triang_masked_softmax_bwd", "softmax_bwd_rowpipe<bf16,causal>",
                  lambda: mfx.mfx_scaled_upper_triang_masked_softmax_bwd(dyc, yc, scale, dx=dxc),
                  4 * valid + 2 * N, N, [], []))
    return [op for op in ops if not only or op.name in only]


def time_isolated(ops, steps, stream, peak):
    out = {}
    for op in ops:
        for _ in range(3):
            op.fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            op.fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        gbs = op.nbytes / (ms * 1e-3) / 1e9
        out[op.name] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac_measured": round(gbs / peak, 4),
                        "elems_per_s": op.elems / (ms * 1e-3), "bytes": op.nbytes}
    return out


# ---------------------------------------------------------------------------
# shape sweep: every op alone on tokens x hidden, bf16 and fp32, with the
# generic path (widths that are not multiples of 8, misaligned pointers), the
# small fp32 case and the fp32 layer shapes; medians of single launches
# ---------------------------------------------------------------------------
L2_BYTES = 129 * 2 ** 20


class L2Flush:
    """Evicts L2 by reading a buffer four times its size (a read leaves clean
    lines, so no write-back of the flush lands inside the next timing)."""

    def __init__(self, dev):
        self.buf = torch.ones(4 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        torch.sum(self.buf, dim=0, out=self.out)


def time_median(fn, reps, stream, flush=None, warm=3):
    """Median over `reps` launches of fn's device time (events on the
    launching stream around each launch; the flush, if any, runs before the
    start event)."""
    for _ in range(warm):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def misalign(t):
    """A copy of t whose data pointer is one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def family_ops(dev, fam, dt, rows, width, misaligned=False, seed=0):
    """The ops of one family on one shape, each with its algorithmic bytes.
    fam: "gelu" (cols = width), "glu" (F = width, input 2F), "dropout"."""
    import elementwise_epilogues_transformer_gb300 as mfx
    from elementwise_epilogues_transformer_gb300 import workloads as W

    s = 2 if dt == torch.bfloat16 else 4
    mis = misalign if misaligned else (lambda t: t)
    ops = []
    if fam == "gelu":
        y, b, g = W.gelu_inputs(rows, width, dt, seed=seed, device=dev)
        y, b, g = mis(y), mis(b), mis(g)
        out = mis(torch.empty_like(y))
        n = rows * width
        ops.append(Op("bias_gelu_fwd", "", lambda: mfx.mfx_bias_gelu_fwd(b, y, out=out),
                      2 * s * n + s * width, n, [], []))
        ops.append(Op("bias_gelu_bwd", "", lambda: mfx.mfx_bias_gelu_bwd(g, b, y, dy=out),
                      3 * s * n + s * width, n, [], []))
    elif fam == "glu":
        x, b, g, w = W.glu_inputs(rows, width, dt, seed=seed, device=dev, with_weight=True)
        x, b, g = mis(x), mis(b), mis(g)
        out = mis(torch.empty(rows, width, dtype=dt, device=dev))
        dx = mis(torch.empty_like(x))
        dw = torch.empty(rows, dtype=torch.float32, device=dev)
        m = rows * width
        fb, bb = 3 * s * m + 2 * s * width, 5 * s * m + 2 * s * width
        ops += [
            Op("bias_geglu_fwd", "", lambda: mfx.mfx_bias_geglu_fwd(x, b, out=out), fb, m, [], []),
            Op("bias_geglu_bwd", "", lambda: mfx.mfx_bias_geglu_bwd(g, x, b, dx=dx), bb, m, [], []),
            Op("bias_swiglu_fwd", "", lambda: mfx.mfx_bias_swiglu_fwd(x, b, out=out), fb, m, [], []),
            Op("bias_swiglu_bwd", "", lambda: mfx.mfx_bias_swiglu_bwd(g, x, b, dx=dx), bb, m, [], []),
            Op("bias_swiglu_w_fwd", "", lambda: mfx.mfx_bias_swiglu_fwd(x, b, w, out=out), fb + 4 * rows,
               m, [], []),
            Op("bias_swiglu_w_bwd", "", lambda: mfx.mfx_bias_swiglu_bwd(g, x, b, w, dx=dx, dweight=dw),
               bb + 8 * rows, m, [], []),
        ]
    else:
        n = rows * width
        x, b, _ = W.dropout_inputs(rows, width, dt, dt, seed=seed, device=dev)
        x, b = mis(x), mis(b)
        out = mis(torch.empty_like(x))
        keep = mis(torch.empty(x.shape, dtype=torch.uint8, device=dev))
        xi = mis(x.clone())
        for rdt in ([dt, torch.float32] if dt == torch.bfloat16 else [dt]):
            r = mis(W.normal((rows, width), rdt, seed + 2, device=dev))
            sr = 2 if rdt == torch.bfloat16 else 4
            tag = "" if rdt == dt else ",res=fp32"
            for p in ((0.0, 0.1, 0.5) if rdt == dt else (0.1,)):
                ops.append(Op(f"bias_dropout_add_train(p={p}{tag})", "",
                              lambda p=p, r=r: mfx.mfx_bias_dropout_add_train(x, b, r, p, 1234, 0, out=out,
                                                                              keep_mask=keep),
                              (2 * s + sr + 1) * n + s * width, n, [], []))
            ops.append(Op(f"bias_dropout_add_inference({tag[1:] or 'res=x'})", "",
                          lambda r=r: mfx.mfx_bias_dropout_add_inference(xi, b, r, 0.1, 1234, 0),
                          (2 * s + sr) * n + s * width, n, [], []))
    return ops


def sweep_entry(ops, reps, stream, peak, flush):
    res = {}
    for op in ops:
        small = op.nbytes < 3 * L2_BYTES
        ms = time_median(op.fn, reps, stream, flush if small else None)
        gbs = op.nbytes / (ms * 1e-3) / 1e9
        res[op.name] = {"ms": round(ms, 4), "gbs": round(gbs, 1), "frac_measured": round(gbs / peak, 4),
                        "frac_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                        "elems_per_s": round(op.elems / (ms * 1e-3)), "l2": "flushed" if small else "> 3x L2"}
    return res


def run_sweep(dev, stream, peak, reps):
    """Every op on the D5 grid (tokens x hidden, bf16 and fp32), plus the
    misaligned-pointer case, the small fp32 case and the fp32 layer shapes.
    One family and shape at a time, so the memory held stays bounded."""
    from elementwise_epilogues_transformer_gb300 import workloads as W

    flush = L2Flush(dev)
    names = {torch.bfloat16: "bf16", torch.float32: "fp32"}
    grid = {}
    for dt in (torch.bfloat16, torch.float32):
        for T in W.SWEEP_TOKENS:
            for H in W.SWEEP_HIDDEN:
                key = f"{names[dt]} T={T} H={H}"
                grid[key] = {}
                for fam in ("gelu", "glu", "dropout"):
                    ops = family_ops(dev, fam, dt, T, H, seed=T + H)
                    grid[key].update(sweep_entry(ops, reps, stream, peak, flush))
                    del ops
                # context, not a library op: torch's own copy of a T x H tensor,
                # timed the same way (at small T launch and latency set the floor)
                src = torch.empty(T, H, dtype=dt, device=dev).normal_()
                dst = torch.empty_like(src)
                ref = [Op("torch_copy_reference", "", lambda: dst.copy_(src), 2 * src.numel() * src.element_size(),
                          src.numel(), [], [])]
                grid[key].update(sweep_entry(ref, reps, stream, peak, flush))
                del ref, src, dst
                torch.cuda.empty_cache()
    special = {}
    for label, fam, dt, T, H, mis in [
            ("misaligned bf16 16384x16384 (every pointer one element off 16 B)", "gelu", torch.bfloat16,
             16384, 16384, True),
            ("misaligned bf16 16384x4096 (every pointer one element off 16 B)", "dropout", torch.bfloat16,
             16384, 4096, True),
            ("misaligned bf16 16384x(2x14336) (every pointer one element off 16 B)", "glu", torch.bfloat16,
             16384, 14336, True),
            ("fp32 1024x4096 (the small fp32 case)", "gelu", torch.float32, 1024, 4096, False),
            ("fp32 16384x16384 (bias-GeLU layer shape)", "gelu", torch.float32, 16384, 16384, False),
            ("fp32 16384x(2x14336) (GLU layer shape)", "glu", torch.float32, 16384, 14336, False),
            ("fp32 [4096x4]x4096 (residual-add layer shape)", "dropout", torch.float32, 16384, 4096, False)]:
        ops = family_ops(dev, fam, dt, T, H, misaligned=mis, seed=7)
        special[label] = sweep_entry(ops, reps, stream, peak, flush)
        del ops
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()

    largest = {k: grid[f"{d} T=65536 H=16384"] for k, d in (("bf16", "bf16"), ("fp32", "fp32"))}
    bf_big = largest["bf16"]
    return {
        "config": ("every op alone on tokens T in {512, 4096, 32768, 65536} x hidden H in {1024, 4096, "
                   "4099, 8192, 16384} (GLU: F = H, input 2F), bf16 and fp32; dropout p in {0, 0.1, "
                   "0.5} with the residual in x's dtype, and p = 0.1 with an fp32 residual for bf16; "
                   f"median of {reps} launches after 3 warm-up; entries under 3x L2 flush L2 (a read of "
                   "4x its size) before each launch; H = 4099 runs the generic path; "
                   "torch_copy_reference is torch's copy of a T x H tensor of the cell's dtype, timed "
                   "the same way, for context (not a library op)"),
        "largest_bf16_min_frac_nominal_8tbs": min(v["frac_nominal_8tbs"] for k, v in bf_big.items()
                                                  if k != "torch_copy_reference"),
        "largest_bf16_min_frac_measured": min(v["frac_measured"] for k, v in bf_big.items()
                                              if k != "torch_copy_reference"),
        "largest": largest,
        "special": special,
        "grid": {k: {op: [v["gbs"], v["frac_measured"]] for op, v in ent.items()} for k, ent in grid.items()},
        "grid_columns": ["GB/s", "fraction of the measured copy peak"],
    }


def host_call_cost(dev, calls=2000):
    """Host cost of one small call: bias-GeLU forward on 512 x 1024 bf16
    issued `calls` times back to back, timed on the host from the first call
    to the end of the last kernel, and on the device between events around
    the loop; through the Python binding, through the C ABI directly
    (ctypes, raw pointers), and torch's own add on the same tensors for
    context.  Where the two times agree the calls are bound by the device,
    where the host time is larger by the host."""
    import elementwise_epilogues_transformer_gb300 as mfx
    from elementwise_epilogues_transformer_gb300 import workloads as W

    y, b, _ = W.gelu_inputs(512, 1024, torch.bfloat16, seed=5, device=dev)
    out = torch.empty_like(y)
    L = mfx.lib()
    st = torch.cuda.current_stream(dev).cuda_stream
    args = (mfx.dtype_code(y.dtype), 512, 1024, b.data_ptr(), y.data_ptr(), out.data_ptr(), st)

    stream = torch.cuda.current_stream(dev)

    def per_call(fn):
        """(host µs per call, device µs per call between events around the loop)"""
        for _ in range(50):
            fn()
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        for _ in range(calls):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        host = 1e6 * (time.perf_counter() - t0) / calls
        return round(host, 2), round(1e3 * a.elapsed_time(e) / calls, 2)

    res = {"workload": "bias_gelu_fwd 512 x 1024 bf16, back to back; each entry [host us per call, "
                       "device us per call]"}
    res["python_binding_us"] = per_call(lambda: mfx.mfx_bias_gelu_fwd(b, y, out=out))
    res["c_abi_us"] = per_call(lambda: L.mfx_bias_gelu_fwd(*args))
    res["torch_add_us"] = per_call(lambda: torch.add(y, b, out=out))
    # the same calls captured once in a CUDA graph and replayed: device time per call
    graph, n = torch.cuda.CUDAGraph(), 100
    with torch.cuda.graph(graph):
        for _ in range(n):
            mfx.mfx_bias_gelu_fwd(b, y, out=out)
    graph.replay()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(calls // n):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    res["cuda_graph_replay_device_us"] = round(1e3 * a.elapsed_time(e) / (n * (calls // n)), 2)
    return res


# ---------------------------------------------------------------------------
# CPU oracle on bounded row samples (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_call(kind, tensors, rows):
    """Run the oracle on the first `rows` rows; return (algorithmic bytes, s)."""
    import oracle as O
    from elementwise_epilogues_transformer_gb300 import workloads as W

    if kind.startswith("gelu"):
        y, b, g = tensors
        yo, bo, go = W.to_oracle(y[:rows]), W.to_oracle(b), W.to_oracle(g[:rows])
        n = yo.size
        t0 = time.perf_counter()
        if kind == "gelu_fwd":
            O.bias_gelu_fwd(yo, bo)
            nb = 4 * n
        else:
            O.bias_gelu_bwd(go, yo, bo)
            nb = 6 * n
        return nb, time.perf_counter() - t0
    if kind.startswith(("geglu", "swiglu")):
        x, b, g, w = tensors
        xo, bo, go = W.to_oracle(x[:rows]), W.to_oracle(b), W.to_oracle(g[:rows])
        wo = W.to_oracle(w[:rows]) if w is not None else None
        m = go.size
        t0 = time.perf_counter()
        if kind == "geglu_fwd":
            O.bias_geglu_fwd(xo, bo)
            nb = 6 * m
        elif kind == "geglu_bwd":
            O.bias_geglu_bwd(go, xo, bo)
            nb = 10 * m
        elif kind == "swiglu_fwd":
            O.bias_swiglu_fwd(xo, bo, wo)
            nb = 6 * m + (4 * rows if wo is not None else 0)
        else:
            O.bias_swiglu_bwd(go, xo, bo, wo)
            nb = 10 * m + (8 * rows if wo is not None else 0)
        return nb, time.perf_counter() - t0
    x, b, r, base = tensors
    xo, bo, ro = W.to_oracle(x[:rows]), W.to_oracle(b), W.to_oracle(r[:rows])
    n = xo.size
    t0 = time.perf_counter()
    if kind == "bda_train":
        O.bias_dropout_add_train(xo, ro, bo, p=0.1, seed=1234, offset=0, elem_base=base)
        nb = 9 * n
    else:
        O.bias_dropout_add_inference(xo, ro, bo)
        nb = 8 * n
    return nb, time.perf_counter() - t0


def oracle_sample(ops, seconds_total):
    """Time the oracle on each op with a row count calibrated so the whole
    sample takes about `seconds_total`; returns (bytes, seconds, description)."""
    per_op = seconds_total / max(1, len(ops))
    tot_b, tot_s, desc = 0, 0.0, []
    for op in ops:
        kind, tensors = op.oracle
        r0 = 2
        nb0, s0 = oracle_call(kind, tensors, r0)
        full = tensors[0].shape[0]
        rows = int(min(full, max(r0, r0 * per_op / max(s0, 1e-6))))
        nb, s = oracle_call(kind, tensors, rows)
        tot_b += nb
        tot_s += s
        desc.append(f"{op.name}:{rows}rows")
    return tot_b, tot_s, desc


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def start_clock_sampler(path):
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader",
                              "-lms", "20"], stdout=f, stderr=subprocess.DEVNULL)
        return p, f
    except (OSError, FileNotFoundError):
        return None, None


def stop_clock_sampler(handle, path, dev_index):
    p, f = handle
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except subprocess.TimeoutExpired:
        p.kill()
    f.close()
    bus = None
    try:
        props = torch.cuda.get_device_properties(dev_index)
        bus = f"{props.pci_bus_id:02X}:{props.pci_device_id:02X}"
    except (AttributeError, RuntimeError):
        pass
    rows = []
    for line in open(path):
        parts = [s.strip() for s in line.split(",")]
        if len(parts) < 10:
            continue
        rows.append(parts)
    if not rows:
        return None
    if bus:
        sel = [r for r in rows if bus in r[1].upper()]
        rows = sel or rows
    if len({r[0] for r in rows}) > 1:
        idx = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[dev_index]
        rows = [r for r in rows if r[0] == idx] or rows

    def mhz(s):
        try:
            return float(s.split()[0])
        except (ValueError, IndexError):
            return None

    sm = [mhz(r[2]) for r in rows if mhz(r[2]) is not None]
    mx = [mhz(r[3]) for r in rows if mhz(r[3]) is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
def source_sha():
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "elementwise_epilogues_transformer_gb300")
    files = sorted(glob.glob(os.path.join(pkg, "csrc", "*"))) + [os.path.join(ROOT, "include", "mfx.h")]
    for fn in files:
        h.update(os.path.basename(fn).encode())
        h.update(open(fn, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(op_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == op_name and parts[1] == sha:
            return float(parts[2])
    return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_reference(args, world, rank):
    """The oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    ops = build_step(dev, 0)
    per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(ops, per_step)
    tb, ts, desc = 0, 0.0, None
    for _ in range(args.steps):
        b, s, desc = oracle_sample(ops, per_step)
        tb += b
        ts += s
    gbs = tb / ts / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * ts / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "row samples per op"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": ", ".join(desc)},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    from elementwise_epilogues_transformer_gb300 import build as B
    if not os.environ.get("MFX_LIBRARY"):
        B.build()
    dev = torch.device("cuda", local if world > 1 else 0)
    global ROWS_SCALE
    ROWS_SCALE = args.rows_scale
    only = tuple(s for s in args.only.split(",") if s)
    next_only = tuple(s for s in args.next_only.split(",") if s)
    ops = build_step(dev, rank, only)
    torch.cuda.synchronize()

    # warm-up
    for _ in range(args.warmup):
        for op in ops:
            op.fn()
    torch.cuda.synchronize()

    # timed region: K steps, events around every launch on the launching stream
    stream = torch.cuda.current_stream(dev)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in ops] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock_path = os.path.join(tempfile.gettempdir(), f"mfx_bench_clocks_{os.getpid()}.csv")
    barrier(world)
    torch.cuda.synchronize()
    sampler = start_clock_sampler(clock_path)
    time.sleep(0.1)
    start.record(stream)
    for k in range(args.steps):
        for i, op in enumerate(ops):
            evs[k][i][0].record(stream)
            op.fn()
            evs[k][i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = stop_clock_sampler(sampler, clock_path, dev.index)
    try:
        os.remove(clock_path)
    except OSError:
        pass

    total_ms = max_over_ranks(start.elapsed_time(end), world)
    step_bytes = sum(op.nbytes for op in ops)
    value = world * step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    per_op = {}
    for i, op in enumerate(ops):
        times = [evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps)]
        ms = sum(times) / args.steps
        gbs = op.nbytes / (ms * 1e-3) / 1e9
        per_op[op.name] = {"ms": round(ms, 4), "ms_median": round(statistics.median(times), 4),
                           "gbs": round(gbs, 1),
                           "frac_measured": round(gbs / peak, 4),
                           "frac_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                           "elems_per_s": op.elems / (ms * 1e-3), "bytes": op.nbytes}
    dom = max(ops, key=lambda o: per_op[o.name]["ms"])
    d = per_op[dom.name]
    roofline = {"bound": "hbm", "kernel": dom.kernel, "op": dom.name, "achieved": d["gbs"],
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(d["gbs"] / peak, 4), "traffic": recorded_traffic(dom.name),
                "algorithmic_bytes": dom.nbytes}

    isolated = None if args.no_isolated else time_isolated(ops, max(args.steps, 20), stream, peak)
    next_ops = None
    if not args.no_next and (not only or next_only):
        del_ops = build_next(dev, next_only)
        next_ops = time_isolated(del_ops, min(args.steps, 100), stream, peak)
        del del_ops
        torch.cuda.empty_cache()

    largest = None
    if args.largest:
        largest = {}
        fams = [("bias_gelu_fwd", "bias_gelu_bwd"),
                ("bias_geglu_fwd", "bias_geglu_bwd", "bias_swiglu_fwd", "bias_swiglu_bwd",
                 "bias_swiglu_w_fwd", "bias_swiglu_w_bwd"),
                ("bias_dropout_add_train", "bias_dropout_add_inference")]
        for fam in fams:   # one family at a time, to bound the memory held
            big_ops = build_step(dev, rank, fam, largest=True)
            res = time_isolated(big_ops, 20, stream, peak)
            for o in big_ops:
                res[o.name]["frac_nominal_8tbs"] = round(res[o.name]["gbs"] / NOMINAL_HBM_GBS, 4)
            largest.update(res)
            del big_ops
            torch.cuda.empty_cache()

    # end to end through the public API with host buffers (before the sweep,
    # whose allocations would otherwise sit in the caching allocator)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(ops, args, world, dev, step_bytes)

    sweep = None
    host_cost = None
    if not args.no_sweep and not only and ROWS_SCALE == 1.0:
        torch.cuda.empty_cache()
        sweep = run_sweep(dev, stream, peak, args.sweep_reps)
        host_cost = host_call_cost(dev)

    cpu = None
    if not args.no_cpu_baseline and world == 1 and rank == 0:
        import multiprocessing
        tb, ts, desc = oracle_sample(ops, args.cpu_seconds)
        cpu = {"value": tb / ts / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "first rows of each op's inputs, " + ", ".join(desc),
               "host_cores_available": multiprocessing.cpu_count()}

    if rank == 0:
        elems = sum(op.elems for op in ops)
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded N(0,1) activations/grads, N(0,0.02) bias, U(0,1) weight)",
                "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (129 MB)",
                           "parallelism": f"replicas x{world} (row shards, no collective)",
                           **({"rows_scale": ROWS_SCALE} if ROWS_SCALE != 1.0 else {})},
                "frac_of_measured_peak": round(value / world / peak, 4),
                "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
                "elements_per_s": world * elems * args.steps / (total_ms * 1e-3),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": len(ops) * args.steps, "clocks": clocks, "per_op": per_op}
        if isolated:
            line["per_op_isolated"] = isolated
        if next_ops:
            line["next_per_op"] = next_ops
        if sweep:
            line["sweep"] = sweep
        if host_cost:
            line["host_call_cost"] = host_cost
        if largest:
            line["largest_per_op"] = {"config": f"{LARGEST['rows']} x {LARGEST['width']} (GLU: F = "
                                                f"{LARGEST['width']}, input 2F wide)", **largest}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(ops, args, world, dev, step_bytes):
    """The step end to end through the public API: every distinct input
    tensor of the step is copied in from pinned host memory and every op's
    outputs are copied back to pinned host memory, inside the timed region.
    Copies run on their own streams (with `--e2e-copy-streams` k > 1,
    tensors of 32 MB and more are split over k streams per direction; on
    GB300 one stream already fills the host link) and overlap the kernels,
    which run on a compute stream, as a caller pipelining the step would; events order every pair of accesses to
    one device buffer (read after write, write after read, write after
    write), across steps too."""
    K = max(1, args.e2e_copy_streams)
    streams = {"compute": torch.cuda.Stream(dev)}
    for k in range(K):
        streams[f"h2d{k}"] = torch.cuda.Stream(dev)
        streams[f"d2h{k}"] = torch.cuda.Stream(dev)
    inputs, seen = [], set()
    for op in ops:
        for t in op.inputs:
            if t is not None and id(t) not in seen:
                seen.add(id(t))
                inputs.append(t)
    host_in = {id(t): torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in inputs}
    host_out = {(i, j): torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for i, op in enumerate(ops) for j, t in enumerate(op.outputs)}
    h2d = sum(t.numel() * t.element_size() for t in inputs)
    d2h = sum(t.numel() * t.element_size() for op in ops for t in op.outputs)
    last_write, last_reads = {}, {}   # id(device tensor) -> [events] / {stream: event}

    def access(parts, reads, writes):
        """Run fn() on each (stream, fn) of `parts`, after every earlier
        conflicting access to the device tensors it reads and writes."""
        deps = [e for t in reads + writes for e in last_write.get(id(t), [])]
        deps += [e for t in writes for e in last_reads.get(id(t), {}).values()]
        evs = {}
        for kind, fn in parts:
            s = streams[kind]
            for e in deps:
                s.wait_event(e)
            with torch.cuda.stream(s):
                fn()
            evs[kind] = torch.cuda.Event()
            evs[kind].record(s)
        for t in reads:
            last_reads.setdefault(id(t), {}).update(evs)
        for t in writes:
            last_write[id(t)] = list(evs.values())
            last_reads[id(t)] = {}

    def copy_parts(direction, dst, src):
        n = dst.numel() * dst.element_size()
        k = K if n >= (32 << 20) else 1
        d, s_ = dst.view(-1).chunk(k), src.view(-1).chunk(k)
        return [(f"{direction}{i}", lambda a=a, b=b: a.copy_(b, non_blocking=True)) for i, (a, b) in enumerate(zip(d, s_))]

    def step():
        for t in inputs:
            access(copy_parts("h2d", t, host_in[id(t)]), [], [t])
        for i, op in enumerate(ops):
            access([("compute", op.fn)], [t for t in op.inputs if t is not None], list(op.outputs))
            for j, t in enumerate(op.outputs):
                access(copy_parts("d2h", host_out[(i, j)], t), [t], [])

    step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        step()
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, world)
    return {"value": round(world * step_bytes * args.e2e_steps / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(1e3 * dt / args.e2e_steps, 3), "steps": args.e2e_steps}


if __name__ == "__main__":
    main()
