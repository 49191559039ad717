"""Build step of libmoe_routing.so (sm_103a only).

Each .cu file under csrc/ is compiled to an object in parallel with nvcc,
then linked into a shared library next to this file. Rebuilds only when a
source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libmoe_routing.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-std=c++17", "-lineinfo",
    # No contraction of separate multiplies and adds: the router's fp32
    # arithmetic must round exactly as written; finalize uses explicit FMAs.
    "-fmad=false",
    "-Xcompiler", "-fPIC", "-I", INCLUDE,
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        name = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(BUILD_DIR, name + ".o")
        log = open(os.path.join(BUILD_DIR, name + ".log"), "w")
        cmd = [nvcc()] + NVCC_FLAGS + ["-Xptxas", "-v", "-c", src, "-o", obj]
        procs.append((name, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    failed = []
    for name, p, log in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append(name)
    if failed:
        msgs = []
        for name in failed:
            with open(os.path.join(BUILD_DIR, name + ".log")) as fh:
                msgs.append(f"--- {name}.cu ---\n" + fh.read()[-4000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run([nvcc()] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
