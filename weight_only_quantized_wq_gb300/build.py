"""Build libwq.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu file under csrc/ is compiled by nvcc in parallel, then linked into
weight_only_quantized_wq_gb300/libwq.so.  No cmake, no torch extension
machinery: the library has no torch dependency.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libwq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


# decode_inst.cu is compiled once per (code width, group schedule) pair; the
# dispatch in decode.cu lists the same pairs.
DECODE_VARIANTS = [(2, 0), (2, 2), (2, 4), (2, -1), (4, 0), (4, 2), (4, -1), (8, 0)]


FLOOR_SRC = os.path.join(PKG, "bench_csrc", "floor.cu")
FLOOR_LIB = os.path.join(PKG, "libwqfloor.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _units():
    """(source, object name, extra flags) for every translation unit."""
    units = []
    for src in _sources():
        base = os.path.basename(src)
        if base == "decode_inst.cu":
            for w, f in DECODE_VARIANTS:
                tag = "w%d_f%s" % (w, "g" if f < 0 else f)
                units.append((src, "decode_inst_%s.o" % tag, ["-DWQ_W=%d" % w, "-DWQ_FOLD=%d" % f]))
        else:
            units.append((src, base + ".o", []))
    return units


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_floor(force: bool = False) -> str:
    """The benchmark's read-only streaming kernel, in a library of its own."""
    if not force and os.path.exists(FLOOR_LIB) and os.path.getmtime(FLOOR_LIB) >= os.path.getmtime(FLOOR_SRC):
        return FLOOR_LIB
    tmp = FLOOR_LIB + ".%d.tmp" % os.getpid()
    r = subprocess.run([nvcc(), *ARCH, *FLAGS, "-shared", "-o", tmp, FLOOR_SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (FLOOR_SRC, r.stdout, r.stderr))
    os.replace(tmp, FLOOR_LIB)
    return FLOOR_LIB


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile and link libwq.so if any source is newer than it (or force)."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = extra or []

    def compile_one(unit):
        src, name, defs = unit
        obj = os.path.join(BUILD, name)
        cmd = [cc, *ARCH, *FLAGS, *defs, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _units()))
    tmp = LIB + ".%d.tmp" % os.getpid()
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None))
