"""Build ``libkvdecode.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` compiles to an object in parallel, then one ``nvcc -shared``
links them with the static CUDA runtime.  No torch headers are involved: the
library's ABI is plain C (``include/kvdecode.h``).

With the environment variable KVD_MARKS=1 the library is built with stage
marks (``-DKVD_MARKS``: the kernels record %globaltimer at numbered points,
read back through kvd_debug_stage_marks; ``bench.py --stage-marks``).  That
build keeps its objects apart and relinks the library whenever the mode
changes; the default build has no marks code at all.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
MARKS = os.environ.get("KVD_MARKS") == "1"
OBJDIR = os.path.join(PKG, "_build_marks" if MARKS else "_build")
LIB = os.path.join(PKG, "libkvdecode.so")
MODE_FILE = os.path.join(PKG, "_build", "library_mode")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC] + (["-DKVD_MARKS"] if MARKS else [])


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(INCLUDE, "kvdecode.h"))
    return hdrs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _mode_changed():
    mode = "marks" if MARKS else "plain"
    try:
        return open(MODE_FILE).read().strip() != mode
    except OSError:
        return True


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OBJDIR, exist_ok=True)
    os.makedirs(os.path.dirname(MODE_FILE), exist_ok=True)
    hdrs = _deps()
    srcs = sources()
    objs = [os.path.join(OBJDIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    jobs = []
    for s, o in zip(srcs, objs):
        if force or ptxas_info or _stale(o, [s] + hdrs):
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", s, "-o", o]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0 or verbose or ptxas_info:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB, objs) or _mode_changed():
        cmd = [nvcc(), *ARCH, "-shared", "-o", LIB + ".tmp", *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(LIB + ".tmp", LIB)
        with open(MODE_FILE, "w") as f:
            f.write("marks" if MARKS else "plain")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv))
