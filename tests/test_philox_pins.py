"""Pins of the oracle's Philox generator (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11).

Both the 32-bit and the 64-bit instances run through one generic round
function in the oracle.  numpy implements Philox4x64-10 independently, so
agreement with numpy checks the round structure (multiplier/word pairing, the
permutation, the key schedule, the round count).  The 32-bit key increments
follow from their definitions; the 32-bit multipliers are the paper's.
"""
import decimal
import math

import numpy as np
import pytest

import oracle as O


@pytest.mark.parametrize("seed", range(6))
def test_philox4x64_matches_numpy(seed):
    rng = np.random.default_rng(seed)
    key = rng.integers(0, 2**64, 2, dtype=np.uint64)
    ctr = rng.integers(0, 2**64, 4, dtype=np.uint64)
    if seed == 0:
        ctr[:] = np.array([2**64 - 1, 5, 0, 0], dtype=np.uint64)
    bg = np.random.Philox(key=key, counter=ctr)
    # numpy advances the 256-bit counter by one before producing each block.
    nxt = ctr.copy()
    for i in range(4):
        nxt[i] = np.uint64((int(nxt[i]) + 1) % 2**64)
        if nxt[i] != 0:
            break
    for _ in range(3):
        ref = bg.random_raw(4)
        assert np.array_equal(O.philox4x64_10(nxt, key), ref)
        for i in range(4):
            nxt[i] = np.uint64((int(nxt[i]) + 1) % 2**64)
            if nxt[i] != 0:
                break


def test_weyl_increments_follow_their_definitions():
    """Two rounds on a zero counter and key expose the key increments:
    round 1 maps zeros to zeros, round 2 xors in the bumped key."""
    out = O.philox4x32_10([0, 0, 0, 0], [0, 0], rounds=2)
    decimal.getcontext().prec = 60
    phi_frac = (decimal.Decimal(5).sqrt() - 1) / 2          # golden ratio - 1
    sqrt3m1 = decimal.Decimal(3).sqrt() - 1
    assert int(out[0]) == int(phi_frac * 2**32)
    assert int(out[2]) == int(sqrt3m1 * 2**32)
    assert out[1] == 0 and out[3] == 0


def test_multipliers_are_the_papers():
    """One round on counter (1, 0, 1, 0) returns the two multipliers as the
    low words: (hi1 ^ 0 ^ 0, lo1, hi0 ^ 0 ^ 0, lo0) = (0, M1, 0, M0)."""
    out = O.philox4x32_10([1, 0, 1, 0], [0, 0], rounds=1)
    assert (int(out[1]), int(out[3])) == (0xCD9E8D57, 0xD2511F53)
    assert out[0] == 0 and out[2] == 0


def test_philox4x32_bit_balance_and_avalanche():
    """Every output bit is balanced over many counters, and flipping one
    counter bit flips about half the output bits (10 rounds mix fully)."""
    n = 4096
    key = [0x12345678, 0x9ABCDEF0]
    outs = np.array([O.philox4x32_10([i, 0, 0, 0], key) for i in range(n)], dtype=np.uint64)
    bits = np.unpackbits(outs.astype(np.uint32).view(np.uint8)).reshape(n, 128)
    p = bits.mean(axis=0)
    assert np.all(np.abs(p - 0.5) < 4 * math.sqrt(0.25 / n) + 0.01)
    flips = []
    for i in range(256):
        a = O.philox4x32_10([i * 977, 3, 5, 7], key)
        b = O.philox4x32_10([i * 977 ^ 1, 3, 5, 7], key)
        flips.append(sum(bin(int(x) ^ int(y)).count("1") for x, y in zip(a, b)))
    assert abs(np.mean(flips) - 64) < 2.0
