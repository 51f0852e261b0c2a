"""Build the native libraries of the package in-tree (nvfp4_skinny_gb300/_build/).

  libnvfp4skinny.so  CUDA kernels + C ABI (include/nvfp4_skinny.h), sm_103a only
  libnvfp4pack.so    host-side NVFP4 packer (include/nvfp4_pack.h), plain C
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "_build")

CUDA_LIB = os.path.join(OUT, "libnvfp4skinny.so")
PACK_LIB = os.path.join(OUT, "libnvfp4pack.so")

CUDA_SOURCES = ["nvfp4_skinny.cu", "quantize.cu", "prefill.cu"]
CUDA_DEPS = ["nvfp4_skinny.cu", "quantize.cu", "prefill.cu", "skinny_kernels.cuh", "gemv_kernels.cuh", "cluster_kernels.cuh",
             "prefill_kernels.cuh",
             "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_cuda(force=False, verbose=False):
    deps = [os.path.join(CSRC, f) for f in CUDA_DEPS] + [os.path.join(INCLUDE, h) for h in ("nvfp4_skinny.h", "nvfp4_prefill.h")]
    if not force and not _stale(CUDA_LIB, deps):
        return CUDA_LIB
    os.makedirs(OUT, exist_ok=True)
    tmp = CUDA_LIB + ".tmp%d" % os.getpid()
    cmd = [_nvcc()] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                              "-cudart", "shared", "-I", INCLUDE, "-o", tmp] + \
          [os.path.join(CSRC, f) for f in CUDA_SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, CUDA_LIB)
    return CUDA_LIB


def build_pack(force=False):
    deps = [os.path.join(CSRC, "nvfp4_pack.c"), os.path.join(INCLUDE, "nvfp4_pack.h")]
    if not force and not _stale(PACK_LIB, deps):
        return PACK_LIB
    os.makedirs(OUT, exist_ok=True)
    tmp = PACK_LIB + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-I", INCLUDE,
                    os.path.join(CSRC, "nvfp4_pack.c"), "-o", tmp, "-lm"], check=True)
    os.replace(tmp, PACK_LIB)
    return PACK_LIB


def build(force=False, verbose=False):
    """Compile both libraries (in parallel); return their paths."""
    with ThreadPoolExecutor(2) as ex:
        fc = ex.submit(build_cuda, force, verbose)
        fp = ex.submit(build_pack, force)
        return fc.result(), fp.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
