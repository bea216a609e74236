"""Build libpkv.so in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_242_gb300.build [--force]

Each translation unit compiles in parallel, then the objects link into
``paged_kv_cache_242_gb300/_build/libpkv.so`` with the CUDA runtime linked
statically and only the ``pkv_*`` symbols exported.

``PKV_NVCC_EXTRA_FLAGS`` (space-separated) adds nvcc options, e.g. the
``-DPKV_*`` tuning definitions of ``csrc/pkv_internal.h`` and
``csrc/decode_stream.cuh``; a build with other flags than the last one
recompiles everything.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libpkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "pkv.h")]


def _flags():
    return NVCC_FLAGS + os.environ.get("PKV_NVCC_EXTRA_FLAGS", "").split()


def _flags_stamp():
    return os.path.join(BUILD_DIR, "flags.txt")


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    try:
        with open(_flags_stamp()) as f:
            if f.read() != " ".join(_flags()):
                return False
    except OSError:
        return False
    built = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(p) <= built for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIBRARY
    nvcc = _nvcc()
    flags = _flags()
    os.makedirs(BUILD_DIR, exist_ok=True)
    objects = []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=8) as pool:
        objects = list(pool.map(compile_one, _sources()))
    version_script = os.path.join(BUILD_DIR, "pkv.map")
    with open(version_script, "w") as f:
        f.write("{ global: pkv_*; local: *; };\n")
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objects + [
        "-Xlinker", f"--version-script={version_script}", "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    with open(_flags_stamp(), "w") as f:
        f.write(" ".join(flags))
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
