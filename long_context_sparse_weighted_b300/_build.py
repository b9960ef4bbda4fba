"""Build liblcsw.so (sm_103a) in-tree with nvcc.

Each .cu under csrc/ is compiled to an object in csrc/../_build/ (parallel,
only when its sources changed), then linked into liblcsw.so next to this file.
"""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblcsw.so")
# the bounds-checked build (-DLCSW_CHECKS=1): same sources, its own objects
OBJ_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "liblcsw_checks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", "-DNDEBUG"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _digest(paths, flags) -> str:
    h = hashlib.sha256()
    for p in sorted(paths):
        with open(p, "rb") as f:
            h.update(p.encode() + f.read())
    h.update(" ".join(ARCH + flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checks: bool = False) -> str:
    """Compile and link liblcsw.so (with checks: liblcsw_checks.so, the
    device-side bounds-checked build); returns its path."""
    obj_dir, lib_path = (OBJ_CHECKS, LIB_CHECKS) if checks else (OBJ, LIB)
    flags = FLAGS + (["-DLCSW_CHECKS=1"] if checks else [])
    os.makedirs(obj_dir, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        stamp = obj + ".sha"
        dig = _digest([src] + headers, flags)
        if not force and not ptxas_info and os.path.exists(obj) and os.path.exists(stamp):
            with open(stamp) as f:
                if f.read() == dig:
                    return obj, False, ""
        cmd = [nvcc, *ARCH, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        with open(stamp, "w") as f:
            f.write(dig)
        return obj, True, r.stderr

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, sources))
    objs = [r[0] for r in results]
    if verbose or ptxas_info:
        for (o, rebuilt, log), src in zip(results, sources):
            if log:
                print(f"== {os.path.basename(src)}\n{log}")
    if force or any(r[1] for r in results) or not os.path.exists(lib_path):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checks="--checks" in sys.argv))
