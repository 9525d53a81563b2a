"""Build libgbscan.so in-tree from csrc/*.cu for sm_103a (GB300).

One translation unit per element type plus the packing kernel and the C ABI,
compiled in parallel with nvcc, then linked into a shared library next to this
file.  No cmake, one -gencode, a minute or so on a 16-core host.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgbscan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libgbscan.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gbscan.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    """Compile (when stale) and return the path of libgbscan.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src):
        obj = os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    srcs = _sources()
    n = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


def ptxas_report(jobs: int | None = None) -> list:
    """Compile every translation unit with -Xptxas -v into a scratch directory (the
    library itself is left alone) and return, per kernel instantiation, what ptxas
    reports: {"unit", "kernel", "registers", "smem", "stack", "spill_stores",
    "spill_loads"}.  This is the compile matrix over element types, operators and
    geometries that the library's kernels are instantiated for."""
    import re
    import tempfile
    cc = nvcc()
    pat_fn = re.compile(r"Compiling entry function '([^']+)'")
    pat_use = re.compile(r"Used (\d+) registers(?:, used \d+ barriers)?(?:, [^,]*?stack size)?(?:, (\d+) bytes smem)?")
    pat_spill = re.compile(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads")
    with tempfile.TemporaryDirectory() as tmp:
        def one(src):
            obj = os.path.join(tmp, os.path.basename(src)[:-3] + ".o")
            r = subprocess.run([cc] + FLAGS + ["-Xptxas", "-v", "-c", src, "-o", obj], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
            rows, cur = [], None
            for line in r.stderr.splitlines():
                m = pat_fn.search(line)
                if m:
                    cur = {"unit": os.path.basename(src), "kernel": m.group(1), "registers": None, "smem": 0,
                           "stack": None, "spill_stores": None, "spill_loads": None}
                    rows.append(cur)
                    continue
                if cur is None:
                    continue
                m = pat_spill.search(line)
                if m:
                    cur["stack"], cur["spill_stores"], cur["spill_loads"] = (int(g) for g in m.groups())
                    continue
                m = pat_use.search(line)
                if m:
                    cur["registers"] = int(m.group(1))
                    cur["smem"] = int(m.group(2) or 0)
            return rows
        srcs = _sources()
        n = jobs or min(len(srcs), os.cpu_count() or 4)
        with cf.ThreadPoolExecutor(max_workers=n) as ex:
            return [row for rows in ex.map(one, srcs) for row in rows]


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
