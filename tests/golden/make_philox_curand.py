"""Writes ``philox4x32_curand.txt``: raw 32-bit words of cuRAND's host
Philox4_32_10 generator, an implementation of Philox4x32-10 (Salmon, Moraes,
Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11) that shares
nothing with this repository.  The words are the known answers the oracle's
Philox4x32-10 is pinned to (``tests/test_philox_pins.py``).

Only cuRAND is called here (through ctypes, on the host: no GPU is needed).
Each line holds a seed, a stream offset and the 16 words the generator emits
from that offset with its default ordering.  Run it from the repository root:

    python tests/golden/make_philox_curand.py
"""
import ctypes
import os

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161   # curandRngType_t in curand.h

# (seed, offset) pairs: zero and full-width seeds (both key words), offsets at
# the start of the stream, inside a block, past the first row of 65536
# subsequences, and far enough out that the counter's high word is nonzero.
CASES = [
    (0, 0),
    (1234, 0),
    (1234, 6),
    (0x0123456789ABCDEF, 0),
    (0x0123456789ABCDEF, 4 * 65536 * 3 + 5),
    (0xFFFFFFFFFFFFFFFF, 1000003),
    (0xDEADBEEF00C0FFEE, 4 * (65536 * (2**32 + 5) + 7) + 2),
    (0x8000000000000001, 2**62 + 9),
]
WORDS = 16


def load_curand():
    names = ["libcurand.so.10", "libcurand.so"]
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    names += [os.path.join(cuda, "lib64", n) for n in ("libcurand.so.10", "libcurand.so")]
    for n in names:
        try:
            return ctypes.CDLL(n)
        except OSError:
            continue
    raise OSError("libcurand not found")


def curand_words(lib, seed, offset, n):
    """n raw words of the host Philox4_32_10 generator from `offset`."""
    gen = ctypes.c_void_p()
    st = lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10)
    if st != 0:
        raise RuntimeError(f"curandCreateGeneratorHost: status {st}")
    try:
        for call, arg in ((lib.curandSetPseudoRandomGeneratorSeed, seed),
                          (lib.curandSetGeneratorOffset, offset)):
            st = call(gen, ctypes.c_ulonglong(arg))
            if st != 0:
                raise RuntimeError(f"{call.__name__}: status {st}")
        buf = (ctypes.c_uint32 * n)()
        st = lib.curandGenerate(gen, buf, ctypes.c_size_t(n))
        if st != 0:
            raise RuntimeError(f"curandGenerate: status {st}")
        return [int(v) for v in buf]
    finally:
        lib.curandDestroyGenerator(gen)


def main():
    lib = load_curand()
    ver = ctypes.c_int()
    lib.curandGetVersion(ctypes.byref(ver))
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "philox4x32_curand.txt")
    with open(out, "w") as f:
        f.write("# Raw 32-bit words of cuRAND's host Philox4_32_10 generator (curand version "
                f"{ver.value}),\n")
        f.write("# default ordering, written by tests/golden/make_philox_curand.py (which calls "
                "only cuRAND).\n")
        f.write("# Columns: seed, offset (in words), then 16 words from that offset, hex.\n")
        for seed, offset in CASES:
            w = curand_words(lib, seed, offset, WORDS)
            f.write(f"{seed:#018x} {offset} " + " ".join(f"{v:08x}" for v in w) + "\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
