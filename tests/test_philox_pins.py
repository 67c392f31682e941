"""Pins of the oracle's Philox generator (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11).

Both the 32-bit and the 64-bit instances run through one generic round
function in the oracle.  numpy implements Philox4x64-10 independently, so
agreement with numpy checks the round structure (multiplier/word pairing, the
permutation, the key schedule, the round count).  The 32-bit key increments
follow from their definitions.  The 32-bit instance as a whole (its
multipliers included) is pinned to cuRAND's host Philox4_32_10 generator,
another independent implementation: stored words in
``tests/golden/philox4x32_curand.txt`` (written by a script that calls only
cuRAND), and a live comparison where libcurand loads.
"""
import decimal
import math
import os

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


# cuRAND's host Philox4_32_10 generator, default ordering, emits its stream as
# 65536 subsequences side by side: word n is word n % 4 of the block with key
# (lo32 seed, hi32 seed) and counter (lo32 i, hi32 i, s, 0), where
# q = n // 4, s = q % 65536 (the subsequence) and i = q // 65536 (the block's
# position in it); the generator offset is the first n.  This layout was
# found by matching the first block of every subsequence, then confirmed at
# every offset below, including ones whose block index needs the counter's
# high word.  Only a generator with the paper's round function, multipliers
# and key schedule reproduces these words.
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_curand.txt")


def _curand_word(n, seed):
    q, k = divmod(n, 4)
    i, s = divmod(q, 65536)
    ctr = [i & 0xFFFFFFFF, i >> 32, s, 0]
    key = [seed & 0xFFFFFFFF, seed >> 32]
    return int(O.philox4x32_10(ctr, key)[k])


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            t = line.split()
            rows.append((int(t[0], 16), int(t[1]), [int(w, 16) for w in t[2:]]))
    return rows


def test_philox4x32_matches_curand_golden_words():
    rows = _golden_rows()
    assert len(rows) == 8 and all(len(w) == 16 for _, _, w in rows)
    assert any(seed >> 32 for seed, _, _ in rows)                 # high key word used
    assert any((off // 4) // 65536 >= 2**32 for _, off, _ in rows)  # high counter word used
    for seed, offset, words in rows:
        got = [_curand_word(offset + j, seed) for j in range(len(words))]
        assert got == words, (hex(seed), offset)


def _load_curand():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_philox_curand", os.path.join(os.path.dirname(__file__), "golden", "make_philox_curand.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    try:
        return mod, mod.load_curand()
    except OSError:
        pytest.skip("libcurand not loadable on this host")


def test_philox4x32_matches_curand_live():
    """Random seeds and offsets (and a run of consecutive words crossing a
    block boundary) drawn from cuRAND's host generator right now."""
    mod, lib = _load_curand()
    rng = np.random.default_rng(77)
    for t in range(12):
        seed = int(rng.integers(0, 2**63)) * 2 + (t & 1)
        offset = int(rng.integers(0, 2**62)) if t % 3 else int(rng.integers(0, 2**20))
        words = mod.curand_words(lib, seed, offset, 10)
        assert words == [_curand_word(offset + j, seed) for j in range(10)], (seed, offset)
