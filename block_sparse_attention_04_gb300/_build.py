"""In-tree build of libmsa.so for sm_103a.

Each .cu is compiled in parallel with nvcc, then linked into one shared
library against the shared CUDA runtime (the one PyTorch already loads).
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(PKG, "_lib", "obj")
LIBMSA = os.path.join(LIBDIR, "libmsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _nvcc():
    p = os.path.join(CUDA_HOME, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + [
        os.path.join(ROOT, "include", "msa.h")]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def link(objs, out, extra=()):
    tmp = out + ".%d.tmp" % os.getpid()
    subprocess.check_call([_nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
                          ["-Xlinker", "-rpath=" + os.path.join(CUDA_HOME, "lib64")] + list(extra))
    os.replace(tmp, out)


def build_libmsa(force=False, verbose=False):
    os.makedirs(OBJDIR, exist_ok=True)
    hdrs = _headers()
    procs, objs = [], []
    for src in _sources():
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJDIR, src[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [_nvcc()] + ARCH + NVCC_FLAGS + ["-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    if force or procs or _stale(LIBMSA, objs):
        link(objs, LIBMSA)
    return LIBMSA


def build(force=False, verbose=False):
    return build_libmsa(force=force, verbose=verbose)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
