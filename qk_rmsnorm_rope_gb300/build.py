"""Build libqknr.so in-tree with nvcc for sm_103a (GB300).

    python -m qk_rmsnorm_rope_gb300.build [--force] [--ptxas-verbose]

Compiles each translation unit of csrc/ in parallel into _build/, then links
the shared library next to this file. No cmake, no JIT: the kernel set is
instantiated ahead of time.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from typing import List

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libqknr.so")
SOURCES = ["qknr_api.cu", "qknr_inst_bf16.cu", "qknr_inst_fp16.cu", "qknr_inst_bf16_early.cu",
           "qknr_inst_fp16_early.cu", "qknr_inst_ring_bf16.cu", "qknr_inst_ring_fp16.cu",
           "qknr_inst_ring_bf16_early.cu", "qknr_inst_ring_fp16_early.cu"]
HEADERS = ["qknr_math.cuh", "qknr_kernel.cuh", "qknr_register_table.cuh", "qknr_ring_kernel.cuh",
           "qknr_ring_table.cuh", "qknr_dispatch.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqknr")
    return path


def _deps() -> List[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(INCLUDE, "qknr.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    if not force and up_to_date():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"--- {src}\n{text}")
        elif text and (ptxas_verbose or not quiet):
            sys.stdout.write(text)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIBRARY + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False))


if __name__ == "__main__":
    main()
