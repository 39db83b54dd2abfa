"""Build libexattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into
``exact_tiled_softmax_gb300/libexattn.so`` with the CUDA runtime linked
statically, so the library depends only on the driver at run time.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libexattn.so")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(nvcc, src, obj, verbose_ptxas):
    cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return res.stderr


def build(verbose_ptxas=False, quiet=True):
    """Compile every kernel source and link libexattn.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(BUILD_DIR, os.path.basename(s)[:-3] + ".o") for s in sources]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        logs = list(ex.map(lambda so: _compile(nvcc, so[0], so[1], verbose_ptxas),
                           zip(sources, objs)))
    if verbose_ptxas and not quiet:
        for src, log in zip(sources, logs):
            print(f"== {os.path.basename(src)}\n{log}")
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv, quiet=False))
