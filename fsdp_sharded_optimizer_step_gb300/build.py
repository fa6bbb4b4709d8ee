"""Builds the CUDA library in-tree: fsdp_sharded_optimizer_step_gb300/_lib/libzero.so.

Device code targets sm_103a only.  Exactness flags: --fmad=false and IEEE
division / square root for the device, -ffp-contract=off for the host code that
derives the binary32 AdamW constants.  The CUDA runtime is linked statically,
so the library loads (and its host-only functions run) without a GPU.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libzero.so")
ROOT = os.path.dirname(HERE)

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-prec-div=true", "-prec-sqrt=true",
              "-Xcompiler", "-fPIC,-ffp-contract=off,-O2", "-Xptxas", "-v"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]

SOURCES_CU = ["zero_kernels.cu", "zero_abi.cu", "zero_noalloc.cu", "zero_reshard.cu"]
SOURCES_CXX = ["zero_plan.cpp", "zero_offload.cpp"]
HEADERS = ["zero_internal.h", "zero_launch.h", "zero_nvtx.h"]
# the host update of the offloaded step: vectorised (-O3; -fno-math-errno lets sqrt
# become one instruction), still one rounding per operation (-ffp-contract=off)
CXX_EXTRA = {"zero_offload.cpp": ["-O3", "-fno-math-errno", "-pthread"]}


def _cuda_include():
    import shutil
    nvcc = shutil.which(NVCC) or NVCC
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")


def _newest_input():
    paths = [os.path.join(CSRC, f) for f in SOURCES_CU + SOURCES_CXX + HEADERS]
    paths.append(os.path.join(ROOT, "include", "zero.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (in parallel) and link the library; returns its path."""
    return _build_into(OUT_DIR, (), force, verbose)


def build_variant(name: str, defines, force: bool = False, verbose: bool = False) -> str:
    """The same library compiled with extra preprocessor definitions (for example
    ZERO_SELFCHECK, the bounds- and alignment-checked diagnostic build) into
    _lib/<name>/libzero.so; returns its path.  The binding loads it instead of the
    normal build when the ZERO_LIB environment variable names it."""
    return _build_into(os.path.join(OUT_DIR, name), tuple(f"-D{d}" for d in defines), force, verbose)


def _build_into(out_dir, defines, force, verbose):
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libzero.so")
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    objs, procs = [], []
    for f in SOURCES_CU:
        o = os.path.join(out_dir, f + ".o")
        cmd = [NVCC, *ARCH, *NVCC_FLAGS, *defines, "-c", os.path.join(CSRC, f), "-o", o]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(o)
    for f in SOURCES_CXX:
        o = os.path.join(out_dir, f + ".o")
        cmd = ["g++", *CXX_FLAGS, *CXX_EXTRA.get(f, []), "-I", _cuda_include(), *defines, "-c",
               os.path.join(CSRC, f), "-o", o]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(o)
    failed = False
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + out)
        failed |= pr.returncode != 0
    if failed:
        raise RuntimeError("building the CUDA library failed (see compiler output above)")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp, "-lpthread", "-ldl"], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
