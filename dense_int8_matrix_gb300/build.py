"""Build libgemm_gb300.so from csrc/ for sm_103a with nvcc (in-tree).

Each translation unit is compiled in parallel into ``_build/`` and linked
into ``libgemm_gb300.so`` beside this file.  The CUDA runtime is linked
statically, so the library depends only on the driver.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgemm_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-v",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        log = obj + ".log"
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        fh = open(log, "w")
        procs.append((subprocess.Popen(cmd, stdout=fh, stderr=subprocess.STDOUT), fh, src, log))
        objs.append(obj)
    failed = []
    for p, fh, src, log in procs:
        rc = p.wait()
        fh.close()
        if rc != 0:
            failed.append((src, log))
        elif verbose:
            sys.stdout.write(open(log).read())
    if failed:
        msgs = []
        for src, log in failed:
            msgs.append("== %s ==\n%s" % (src, open(log).read()))
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    link = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
