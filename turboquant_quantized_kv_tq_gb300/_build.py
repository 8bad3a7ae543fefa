"""Build the C-ABI library ``libtq.so`` in-tree for sm_103a (GB300).

Each translation unit is compiled in parallel with nvcc (CUDA sources) or g++ (host sources),
then linked into ``turboquant_quantized_kv_tq_gb300/_lib/libtq.so`` with the CUDA runtime linked
statically.  Objects go to ``_build/`` at the repository root.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtq.so")
OBJ_DIR = os.path.join(ROOT, "_build", "obj")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(src, extra_nvcc=()):
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    out = os.path.join(OBJ_DIR, src + ".o")
    path = os.path.join(CSRC, src)
    if src.endswith(".cu"):
        cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-ffp-contract=off",
               "-I", INCLUDE, "-I", CSRC, *extra_nvcc, "-c", path, "-o", out]
    else:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC,
               "-I", os.path.join(cuda, "include"), "-c", path, "-o", out]
    res = subprocess.run(cmd, capture_output=True, text=True)
    return src, res.returncode, res.stdout + res.stderr, out


def build(verbose=False, extra_nvcc=()):
    """Compile every source and link libtq.so; raise RuntimeError on the first failure."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra_nvcc), srcs))
    objs = []
    for src, rc, log, out in results:
        if verbose and log.strip():
            print(f"[{src}]\n{log}", file=sys.stderr)
        if rc != 0:
            raise RuntimeError(f"compiling {src} failed:\n{log}")
        objs.append(out)
    cuda = _cuda_home()
    tmp = LIB_PATH + ".tmp"
    cmd = [os.path.join(cuda, "bin", "nvcc"), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("linking libtq.so failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
