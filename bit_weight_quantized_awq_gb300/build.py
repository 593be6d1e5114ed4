"""Builds the library ``_build/libawq_gb300.so`` in-tree with nvcc for sm_103a.

Every ``csrc/*.cu`` translation unit is compiled in parallel, then linked
into one shared library with the CUDA runtime linked statically. Rebuilds
only what is older than its sources (any header change rebuilds all units).

It also builds ``_build/libawq_gb300_fault_test.so``, the fault-test build
used only by the tests: the units with bounded device waits (the C ABI, the
decode and prefill kernels) compiled again with ``-DAWQ_FAULT_TEST`` (a wait
limit of about 2 ms and the switch declared in
``include/awq_gb300_fault_test.h``), linked with the other units' objects.

    python -m bit_weight_quantized_awq_gb300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libawq_gb300.so")
FAULT_LIB = os.path.join(BUILD, "libawq_gb300_fault_test.so")
FAULT_BUILD = os.path.join(BUILD, "fault_test")
# units whose kernels wait on barriers or flags (and the ABI that sets the switch)
FAULT_UNITS = ("awq_api.cu", "awq_decode.cu", "awq_prefill.cu")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the AWQ library needs the CUDA toolkit to build")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _fault_obj(src: str) -> str:
    return os.path.join(FAULT_BUILD, os.path.basename(src)[:-3] + ".o")


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(FAULT_BUILD, exist_ok=True)
    cc = nvcc()
    headers = _headers()
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers + [os.path.abspath(__file__)]):
            cmd = [cc] + ARCH + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_verbose else []) + \
                  ["-c", src, "-o", obj]
            jobs.append((src, cmd))
        if os.path.basename(src) in FAULT_UNITS:
            fobj = _fault_obj(src)
            if force or _stale(fobj, [src] + headers + [os.path.abspath(__file__)]):
                jobs.append((src + " (fault test)", [cc] + ARCH + NVCC_FLAGS + ["-DAWQ_FAULT_TEST", "-c", src,
                                                                               "-o", fobj]))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in _sources()]
    fault_objs = [_fault_obj(s) if os.path.basename(s) in FAULT_UNITS else
                  os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in _sources()]

    def run(job):
        src, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    failed = []
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, r in ex.map(run, jobs):
                if r.returncode != 0:
                    failed.append((src, r.stderr))
                elif (ptxas_verbose or r.stderr.strip()) and not quiet:
                    sys.stderr.write(r.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{e}" for s, e in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    for lib, lib_objs in ((LIB, objs), (FAULT_LIB, fault_objs)):
        if force or jobs or _stale(lib, lib_objs):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [cc] + ARCH + ["-shared", "-o", tmp] + lib_objs
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose))
