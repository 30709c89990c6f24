"""Build libloong_attn.so in-tree with nvcc for sm_103a.

Compiles every ``csrc/*.cu`` in parallel (one process per translation unit)
and links them into ``head_context_attention_gb300/libloong_attn.so`` with the
CUDA runtime linked statically, so the library needs no CUDA shared library
at load time (the driver is opened on first use).  The same sources are also
built with ``-DLOONG_CHECKED`` into ``libloong_attn_checked.so``: every TMA
coordinate, bulk-copy range and plain global store is checked against its
tensor on the device, a failed check sets the device error word (reported as
LOONG_ERR_DEVICE_CHECK) and the store is skipped.
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libloong_attn.so")
LIB_CHECKED = os.path.join(PKG, "libloong_attn_checked.so")
VARIANTS = ((LIB, "", []), (LIB_CHECKED, "checked.", ["-DLOONG_CHECKED"]))
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
    if not all(os.path.exists(lib) for lib, _, _ in VARIANTS):
        return True
    t = min(os.path.getmtime(lib) for lib, _, _ in VARIANTS)
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(PKG, "..", "include", "loong_attn.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force=False, verbose=False):
    """Build both variants; returns the path of the regular library."""
    srcs = sources()
    if not force and not _stale(srcs):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    procs = []
    for lib, tag, extra in VARIANTS:
        for s in srcs:
            base = os.path.join(BUILD, tag + os.path.basename(s))
            log = open(base + ".log", "w")
            cmd = [nv, *ARCH, *FLAGS, *extra, "-I", os.path.join(PKG, "..", "include"), "-c", s, "-o", base + ".o"]
            procs.append((lib, base, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    objs, failed = {lib: [] for lib, _, _ in VARIANTS}, []
    for lib, base, log, p in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(base)
        objs[lib].append(base + ".o")
    if failed:
        msgs = []
        for base in failed:
            with open(base + ".log") as f:
                msgs.append(f"--- {os.path.basename(base)}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    for lib, _, _ in VARIANTS:
        tmp = lib + ".tmp"
        cmd = [nv, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs[lib]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, lib)
    if verbose:
        for s in srcs:
            with open(os.path.join(BUILD, os.path.basename(s) + ".log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
