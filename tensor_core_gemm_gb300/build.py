"""Build libmk.so in-tree: the C-ABI host compiler/runtime (C++) and the sm_103a megakernel.

    python -m tensor_core_gemm_gb300.build        # or tensor_core_gemm_gb300.build.build()

Translation units compile in parallel (nvcc for the kernel, g++ for the host code) and link
with nvcc against the static CUDA runtime. Only sm_103a is generated.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmk.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return cmd, r.returncode, r.stdout


def build(verbose=False, ptxas_verbose=False):
    """Compile every source and link libmk.so; raises RuntimeError with the compiler output."""
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    common_inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include")]
    jobs = []
    objs = []
    for name in sorted(os.listdir(CSRC)):
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name + ".o")
        if name.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   *common_inc, "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
        elif name.endswith(".cpp"):
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function",
                   *common_inc, "-c", src, "-o", obj]
        else:
            continue
        jobs.append(cmd)
        objs.append(obj)
    with ThreadPoolExecutor(max_workers=max(2, len(jobs))) as ex:
        results = list(ex.map(_run, jobs))
    failed = [(c, out) for c, rc, out in results if rc != 0]
    if verbose or ptxas_verbose:
        for c, rc, out in results:
            if out.strip():
                print(" ".join(c[-3:]), "\n", out)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + out for c, out in failed)
        raise RuntimeError("libmk build failed:\n" + msg)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    _, rc, out = _run(cmd)
    if rc != 0:
        raise RuntimeError("libmk link failed:\n" + " ".join(cmd) + "\n" + out)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    path = build(verbose=True, ptxas_verbose="-v" in sys.argv)
    print("built", path)
