"""Build libreplayssm.so in-tree with nvcc for sm_103a (GB300).

The translation units compile in parallel into ``_build/<machine>/`` and link
into ``libreplayssm.so`` next to this file.  A stamp of the sources, flags,
compiler version and host machine decides whether a rebuild is needed, so an
x86 build never gets reused on an Arm host or the reverse.
"""

import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libreplayssm.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

SOURCES = ["abi.cu", "mamba2.cu", "mamba2_variants.cu", "mamba2_f32in.cu", "gdn.cu", "conventional.cu", "materialize.cu", "materialize_pipe.cu", "spec.cu", "spec_tc.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "launch.h", "mamba2.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the ReplaySSM library needs the CUDA toolkit to build")


def _stamp(nvcc):
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "replayssm.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    h.update(platform.machine().encode())
    h.update(subprocess.run([nvcc, "--version"], capture_output=True, text=True).stdout.encode())
    return h.hexdigest()


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link the library if it is missing or out of date.

    Returns the path of the shared library.  ``ptxas_info`` prints register,
    spill and shared-memory figures per kernel (-Xptxas -v).
    """
    nvcc = _nvcc()
    bdir = os.path.join(HERE, "_build", platform.machine())
    os.makedirs(bdir, exist_ok=True)
    stamp = _stamp(nvcc)
    stamp_file = os.path.join(bdir, "stamp")
    if not force and not ptxas_info and os.path.exists(LIB_PATH) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB_PATH
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src} ---\n{out}")
        elif (verbose or ptxas_info) and out:
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
