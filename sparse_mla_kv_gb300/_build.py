"""Build libhs.so in-tree with nvcc for sm_103a (no cmake; translation units compiled in parallel).

build(variant="checked") builds the bounds-checked library, libhs_checked.so (HS_CHECKED=1), into its
own object folder."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhs.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


VARIANTS = {"": (), "checked": ("-DHS_CHECKED=1",)}


def lib_path(variant: str = "") -> str:
    """The shared library of a build variant: libhs.so, or libhs_<variant>.so (e.g. the bounds-checked
    build, compiled with HS_CHECKED=1)."""
    return LIB if not variant else os.path.join(HERE, f"libhs_{variant}.so")


def build(force: bool = False, verbose: bool = False, extra: tuple = (), variant: str = "") -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown build variant {variant!r}")
    extra = tuple(extra) + VARIANTS[variant]
    lib_out = lib_path(variant)
    bdir = BUILD if not variant else os.path.join(BUILD, variant)
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h")))
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(bdir, os.path.basename(s).replace(".", "_") + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([NVCC, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            print(" ".join(cmd))
            print(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib_out, objs):
        run([NVCC, *ARCH, "-shared", "-o", lib_out, *objs])
    return lib_out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=tuple(a for a in sys.argv[1:] if a.startswith("-X")),
                variant="checked" if "--checked" in sys.argv else ""))
