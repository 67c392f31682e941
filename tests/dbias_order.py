"""The summation order of the fused bias gradients, restated for the tests.

Every fused backward with a bias gradient (include/mfx.h, the `*_dbias`
calls) sums the gradient *as stored* (rounded to its dtype) over rows in two
fixed stages, whichever kernel produced the gradient:

1. J partial sums per column: partial j adds rows j, j + J, j + 2J, ... in
   increasing row order into an fp32 accumulator that starts at 0.  They land
   in the workspace as a [J, W] fp32 array (row j = partial j).
2. One finishing pass per column: 32 warps; warp w adds partials
   j = w + 32 k + 256 m (k = 0..7, m = 0, 1, ...) into eight accumulators
   a[k] in increasing m; the eight are added pairwise,
   ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)); the 32 warp sums go
   round-robin into four accumulators s[w mod 4] in warp order, and the
   result (s0 + s1) + (s2 + s3) is rounded once to the bias dtype.

J is the kernel's choice (it follows the launch grid), so the tests read it
off the workspace: filled with NaN before the call, exactly its first J rows
are overwritten.  Given J, `replay` repeats both stages in numpy float32
(IEEE single additions, round to nearest even), so a kernel that dropped,
doubled or misplaced a single term would not reproduce its bits;
`tolerance` gives the classical error bound of that order against the exact sum of the
stored values (every term passes through at most `depth` fp32 additions).
"""
import math

import numpy as np
import torch

FINISH_WARPS = 32
U = 2.0 ** -24  # fp32 unit roundoff


def nan_workspace(nbytes, device):
    """A workspace whose every fp32 word is a NaN (all bits set)."""
    return torch.full((max(int(nbytes), 16),), 0xFF, dtype=torch.uint8, device=device)


def partials_written(ws, W):
    """J: the number of leading [W]-rows of the fp32 workspace the call
    overwrote (the rest still hold the NaN fill)."""
    n = ws.numel() // 4 // W
    rows = ws[: n * W * 4].view(torch.float32).view(n, W).cpu().numpy()
    written = ~np.isnan(rows).all(axis=1)
    J = int(np.argmin(written)) if not written.all() else n
    assert written[:J].all() and not written[J:].any(), "partials must be a leading block of rows"
    assert not np.isnan(rows[:J]).any(), "every written partial row is complete"
    return J


def replay(stored, J):
    """Both stages on `stored` (float32 [rows, W]) with J partials; float32 [W]."""
    stored = np.ascontiguousarray(stored, dtype=np.float32)
    rows, W = stored.shape
    part = np.zeros((J, W), dtype=np.float32)
    for r0 in range(0, rows, J):
        blk = stored[r0:r0 + J]
        part[: blk.shape[0]] += blk
    warp = np.zeros((FINISH_WARPS, W), dtype=np.float32)
    step = 8 * FINISH_WARPS
    for w in range(FINISH_WARPS):
        a = np.zeros((8, W), dtype=np.float32)
        j = w
        while j + 7 * FINISH_WARPS < J:
            for k in range(8):
                a[k] += part[j + k * FINISH_WARPS]
            j += step
        for k in range(7):
            if j + k * FINISH_WARPS < J:
                a[k] += part[j + k * FINISH_WARPS]
        warp[w] = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]))
    s = np.zeros((4, W), dtype=np.float32)
    for w in range(FINISH_WARPS):
        s[w & 3] += warp[w]
    return (s[0] + s[1]) + (s[2] + s[3])


def round_to(v32, dtype):
    """float32 values rounded to the bias dtype (RNE), as float64."""
    return torch.from_numpy(np.asarray(v32, dtype=np.float32)).to(dtype).double().numpy()


def depth(rows, J):
    """Most fp32 additions any term passes through: its partial (at most
    ceil(rows / J) terms), its finishing accumulator (ceil(J / 256)), the
    pairwise eight (3), the round-robin warp sums (8) and the last pair (2)."""
    return math.ceil(rows / J) + math.ceil(J / (8 * FINISH_WARPS)) + 3 + FINISH_WARPS // 4 + 2


def column_sums(stored):
    """Exact-enough float64 sums and sums of magnitudes per column of a
    [rows, W] array, in row chunks (bounded host memory)."""
    rows, W = stored.shape
    s = np.zeros(W, dtype=np.float64)
    a = np.zeros(W, dtype=np.float64)
    for r0 in range(0, rows, 1024):
        blk = np.asarray(stored[r0:r0 + 1024], dtype=np.float64)
        s += blk.sum(axis=0)
        a += np.abs(blk).sum(axis=0)
    return s, a


def tolerance(got, exact, abs_sum, rows, J, bf16):
    """|dbias - exact| allowed by the order: gamma_d * sum|terms| (d = depth)
    for the fp32 stages, plus half a bf16 ulp for the final rounding when the
    bias is bf16 (at the larger of the two magnitudes), plus the float64
    reference's own rounding (rows * 2^-53 * sum|terms|)."""
    from parity import bf16_ulp
    d = depth(rows, J)
    tol = (d * U / (1.0 - d * U) + rows * 2.0 ** -53) * abs_sum
    if bf16:
        tol = tol + 0.5 * bf16_ulp(np.maximum(np.abs(got), np.abs(exact)))
    return tol
