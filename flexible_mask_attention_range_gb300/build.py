"""In-tree build of libffa.so (the C-ABI library) for sm_103a with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into one shared object next
to this file.  Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libffa.so")
SOURCES = ["ffa_api.cu", "ffa_plan.cu", "ffa_fwd.cu", "ffa_bwd.cu", "ffa_noalloc.cu", "ffa_decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libffa.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def check_forward_registers(ptxas_log: str) -> None:
    """The forward kernel rebalances registers between warpgroups (setmaxnreg); the split in
    its source is exact for one launch register count (kRegsLaunch).  Refuse a build whose
    forward kernels were given any other count: such a launch could wait forever."""
    src = open(os.path.join(CSRC, "ffa_fwd.cu")).read()
    want = int(re.search(r"kRegsLaunch = (\d+)", src).group(1))
    found = []
    current = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current is not None:
            if "ffa_fwd_kernel" in current:
                found.append(int(m.group(1)))
            current = None
    if not found:
        raise RuntimeError("no register report for the forward kernels in the ptxas output")
    bad = [n for n in found if n != want]
    if bad:
        raise RuntimeError(f"forward kernels built with {sorted(set(bad))} registers per thread; the register "
                           f"split needs exactly {want}")


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        extra = ["-Xptxas", "-v"] if src == "ffa_fwd.cu" and not ptxas_info else []
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + flags + extra
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        log = r.stdout + r.stderr
        if src == "ffa_fwd.cu":
            check_forward_registers(log)
        return obj, log if (verbose or ptxas_info or not extra) else ""

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [cc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + ["-lcudart_static", "-lrt", "-ldl",
                                                                          "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def ensure_built() -> str:
    if needs_build():
        build()
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
