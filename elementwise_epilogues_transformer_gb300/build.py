"""Build ``libmfx.so`` in-tree for GB300 (sm_103a) with nvcc.

Each CUDA translation unit is compiled on its own (in parallel) and the
objects are linked into one shared library with the CUDA runtime linked
statically, so the library only needs the driver at run time.  No fast-math
flags: the fp32 paths rely on IEEE division and libdevice ``expf``, and the
dropout path on explicit round-to-nearest intrinsics.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmfx.so")

SOURCES = ["mfx_abi.cu", "gelu.cu", "glu.cu", "dropout.cu", "dbias.cu", "sqrelu.cu", "softmax.cu"]
HEADERS = ["mfx_device.cuh", "mfx_host.h", "mfx_pipe.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmfx")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), lib=None, build_dir=None) -> str:
    """Compile (if needed) and return the path of libmfx.so.

    `defines` (e.g. ["MFX_PREFETCH=0"]) override the kernels' compile-time
    tuning knobs; with them, give `lib` and `build_dir` for the variant."""
    LIB = lib or globals()["LIB"]
    BUILD = build_dir or globals()["BUILD"]
    flags = [*NVCC_FLAGS, *(f"-D{d}" for d in defines)]
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "mfx.h"),
                                                           os.path.abspath(__file__)]
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [nvcc(), *flags, "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        log = os.path.join(BUILD, os.path.basename(o) + ".ptxas.txt")
        with open(log, "w") as f:
            f.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {s}:\n{r.stderr[-4000:]}")
        return o

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
    if verbose:
        for src in SOURCES:
            print(open(os.path.join(BUILD, src.replace(".cu", ".o") + ".ptxas.txt")).read())
    return LIB


if __name__ == "__main__":
    print(build(force=True))
