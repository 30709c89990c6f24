"""Build libloong_attn.so in-tree with nvcc for sm_103a.

Compiles every ``csrc/*.cu`` in parallel (one process per translation unit)
and links them into ``head_context_attention_gb300/libloong_attn.so`` with the
CUDA runtime linked statically, so the library needs no CUDA shared library
at load time (the driver is opened on first use).
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libloong_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(srcs):
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(PKG, "..", "include", "loong_attn.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force=False, verbose=False):
    srcs = sources()
    if not force and not _stale(srcs):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    procs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s) + ".o")
        log = open(os.path.join(BUILD, os.path.basename(s) + ".log"), "w")
        cmd = [nv, *ARCH, *FLAGS, "-I", os.path.join(PKG, "..", "include"), "-c", s, "-o", obj]
        procs.append((s, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    objs, failed = [], []
    for s, obj, log, p in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(s)
        objs.append(obj)
    if failed:
        msgs = []
        for s in failed:
            with open(os.path.join(BUILD, os.path.basename(s) + ".log")) as f:
                msgs.append(f"--- {os.path.basename(s)}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + ".tmp"
    cmd = [nv, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    if verbose:
        for s in srcs:
            with open(os.path.join(BUILD, os.path.basename(s) + ".log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
