"""Build the CUDA library libpkv.so in-tree (paged_kv_cache_215_gb300/_build/).

Each .cu file is compiled by nvcc for sm_103a in parallel, the host C++ file by
g++, and the objects are linked into one shared library against the CUDA
runtime.  No CMake, no setuptools: one nvcc invocation per translation unit.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(BUILD, "libpkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _sources():
    cus = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cpps = sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = cus + cpps + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return cus, cpps, deps


def _stale(deps) -> bool:
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    return any(os.path.getmtime(d) > t for d in deps + [__file__])


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    cus, cpps, deps = _sources()
    if not force and not _stale(deps):
        return SO
    os.makedirs(BUILD, exist_ok=True)
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include")]
    jobs = []
    for src in cus:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-fvisibility=hidden", *inc, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    for src in cpps:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", *inc, "-c", src,
               "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        for l in logs:
            if l.strip():
                print(l)
    tmp = SO + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs],
          "-L", os.path.join(cuda, "lib64"), "-lcudart",
          "-Xlinker", "-rpath=" + os.path.join(cuda, "lib64")])
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
