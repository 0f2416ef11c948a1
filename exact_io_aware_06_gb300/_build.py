"""Build libfa.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file compiles to an object in parallel; the objects link into
``exact_io_aware_06_gb300/_lib/libfa.so`` with the CUDA runtime linked
statically, so the library needs no driver at load time (the driver is
reached through the runtime's entry-point query when a kernel launches).
A stamp file holding a hash of the sources and flags skips up-to-date builds.
"""
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB = os.path.join(OUT_DIR, "libfa.so")
STAMP = os.path.join(OUT_DIR, "libfa.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(extra_flags):
    h = hashlib.sha256()
    for path in sorted(sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                    if f.endswith((".h", ".cuh"))] +
                       [os.path.join(INCLUDE, "fa.h")]):
        h.update(path.encode())
        with open(path, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def up_to_date(extra_flags=()):
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as fh:
        return fh.read().strip() == _digest(extra_flags)


def build(verbose=False, extra_flags=()):
    """Compile and link; returns the library path.  Raises on failure."""
    if up_to_date(extra_flags):
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    exe = nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [exe] + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if verbose and text:
            sys.stdout.write(text)
        if p.returncode != 0:
            failed.append((src, text))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"{s}:\n{t}" for s, t in failed))
    tmp = LIB + ".tmp"
    link = [exe] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    p = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n" + p.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as fh:
        fh.write(_digest(extra_flags))
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
