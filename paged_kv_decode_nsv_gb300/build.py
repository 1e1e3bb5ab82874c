"""Build libnsv.so (the C-ABI library) for sm_103a with nvcc.

Each .cu file compiles in parallel into _build/, then one link makes
paged_kv_decode_nsv_gb300/_lib/libnsv.so against the shared CUDA runtime (the
same libcudart.so a PyTorch process already holds, so streams and the device
context are shared).  Run ``python -m paged_kv_decode_nsv_gb300.build``
(``--force`` to rebuild, ``--ptxas`` to print register and spill counts).
"""

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libnsv.so")
SOURCES = ["nsv_api.cu", "decode.cu", "kv_write.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def cuda_home():
    return os.path.dirname(os.path.dirname(os.path.realpath(_nvcc())))


def compile_flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
                   "-Xcompiler", "-fPIC,-fvisibility=hidden", *extra]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link libnsv.so; returns its path."""
    if not force and not ptxas_info and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + compile_flags(extra)
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif text.strip() and (verbose or ptxas_info):
            print(text, flush=True)
    if failed:
        msg = "\n".join("== %s ==\n%s" % f for f in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB + ".tmp.%d" % os.getpid()
    rpath = os.path.join(cuda_home(), "lib64")
    cmd = [nvcc, "-shared", "-cudart", "shared"] + ARCH + ["-o", tmp] + objs + \
          ["-Xlinker", "-rpath," + rpath]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv))
