"""Build the CUDA shared library ``_lib/libqgemv.so`` in-tree (sm_103a only).

Compiles the per-format kernel units, the expert kernels, the C ABI and the host
packer in parallel with nvcc / g++, then links one shared library.  Object files go to
``_build/`` at the repository root.  A stamp of the sources and flags skips
the work when nothing changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libqgemv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "-I", INCLUDE, "-I", CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-I", INCLUDE, "-I", CSRC]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _units():
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    cxx = os.environ.get("CXX", "g++")
    units = []
    for f in range(5):
        units.append((os.path.join(BUILD, f"qgemv_inst_fmt{f}.o"),
                      [nvcc, *ARCH, *NVCC_FLAGS, f"-DQG_INST_FMT={f}", "-c",
                       os.path.join(CSRC, "qgemv_inst.cu")]))
    units.append((os.path.join(BUILD, "qgemv_experts.o"),
                  [nvcc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, "qgemv_experts.cu")]))
    units.append((os.path.join(BUILD, "qgemv_api.o"),
                  [nvcc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, "qgemv_api.cu")]))
    for src in ("pack.cpp", "tile_select.cpp"):
        units.append((os.path.join(BUILD, src.replace(".cpp", ".o")),
                      [cxx, *CXX_FLAGS, "-c", os.path.join(CSRC, src)]))
    return cuda, nvcc, units


def _stamp(cmds) -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["qgemv.h"]
    for name in files:
        path = os.path.join(CSRC, name) if name != "qgemv.h" else os.path.join(INCLUDE, name)
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as fh:
                h.update(fh.read())
    h.update(repr(cmds).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link; return the path of the shared library."""
    cuda, nvcc, units = _units()
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", LIB, *[o for o, _ in units],
            "-Xlinker", f"-rpath,{os.path.join(cuda, 'lib64')}", "-lpthread"]
    stamp = _stamp([c for _, c in units] + [link])
    stamp_file = os.path.join(BUILD, "libqgemv.stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as fh:
            if fh.read().strip() == stamp:
                return LIB

    def run(unit):
        out, cmd = unit
        full = cmd + ["-o", out]
        if verbose:
            print(" ".join(full), flush=True)
        r = subprocess.run(full, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(full)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max_workers=min(len(units), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(run, units))
    if verbose:
        for log in logs:
            if log.strip():
                print(log)
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}\n{r.stderr}")
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
