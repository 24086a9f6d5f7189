"""Build libsamspec.so in-tree for sm_103a (nvcc, one -gencode, translation
units compiled in parallel, then linked), and the debug library
libsamspec_checks.so (-DSAMSPEC_CHECKS=1: every automaton index checked
against its array)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsamspec.so")
CHECKS_LIB = os.path.join(OUT_DIR, "libsamspec_checks.so")
SOURCES = ["abi.cu", "sam.cu", "sampling.cu", "verify.cu"]
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags():
    return ["-O3", "-std=c++17", "-lineinfo", "-gencode", GENCODE, "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, "--expt-relaxed-constexpr"]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


CHECKED_SOURCES = ["sam.cu"]  # the only translation unit SAMSPEC_CHECKS changes


def _jobs(checks: bool, force: bool, ptxas_info: bool):
    """(objects, link target, compile commands still needed) of one library;
    the debug library shares every object but the checked ones."""
    nvcc = nvcc_path()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "samspec.h"))
    objs, cmds = [], []
    for src in SOURCES:
        checked = checks and src in CHECKED_SOURCES
        obj_dir = OBJ_DIR + ("_checks" if checked else "")
        os.makedirs(obj_dir, exist_ok=True)
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if (checked or not checks) and (force or _stale(o, [s] + headers)):
            cmds.append([nvcc] + _flags() + (["-DSAMSPEC_CHECKS=1"] if checked else []) +
                        (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", s, "-o", o])
    return objs, (CHECKS_LIB if checks else LIB), cmds


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checks: bool = True) -> str:
    """Compiles the library (and, with checks, the debug library) if a source
    changed; returns the library's path."""
    nvcc = nvcc_path()
    os.makedirs(OUT_DIR, exist_ok=True)
    libs = [_jobs(False, force, ptxas_info)] + ([_jobs(True, force, ptxas_info)] if checks else [])
    jobs = [c for _, _, cmds in libs for c in cmds]
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
                if verbose or ptxas_info or res.returncode != 0:
                    print(" ".join(cmd))
                    print(res.stdout + res.stderr)
                if res.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{res.stderr}")
    for objs, lib, _ in libs:
        if force or _stale(lib, objs):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc, "-shared", "-gencode", GENCODE, "--cudart", "static", "-o", tmp] + objs
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"link failed: {' '.join(cmd)}\n{res.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
