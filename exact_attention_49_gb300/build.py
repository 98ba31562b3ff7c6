"""Build the CUDA library ``libfa49.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in ``_build/`` in parallel
(``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``) and the
objects are linked into ``exact_attention_49_gb300/libfa49.so``.  ptxas
resource usage (registers, spills, shared memory) is written to
``_build/ptxas.log``.  The CUDA runtime is linked statically; the driver entry
point for tensor maps is looked up at run time, so no libcuda link is needed.
"""
from __future__ import annotations

import glob
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa49.so")
ROOT = os.path.dirname(PKG)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _sources() + _headers() + [__file__])


def ptxas_report(text: str) -> dict:
    """Per kernel (mangled name): registers, spill stores and spill loads, from ptxas -v output."""
    out = {}
    cur = None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            out[cur] = {"registers": None, "spill_stores": 0, "spill_loads": 0}
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            out[cur]["spill_stores"], out[cur]["spill_loads"] = int(m.group(1)), int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            out[cur]["registers"] = int(m.group(1))
    return out


# The forward kernel splits its registers between warpgroups with setmaxnreg, assuming it is
# launched at exactly this many registers per thread (FwdCfg::REG_LAUNCH): an increase beyond
# what the launch holds would wait forever, so the build refuses any other count.
FWD_LAUNCH_REGISTERS = 168


# The forward's decoding configuration (template flag DEC, mangled "ELb1E") runs two CTAs of
# 192 threads per SM with no split: it only has to fit under the same count.
FWD_DECODING = re.compile(r"fwd_kernelILi\d+ELi\d+ELb1E")


def check_register_split(report: dict) -> None:
    for name, r in report.items():
        if FWD_DECODING.search(name):
            if r["registers"] > FWD_LAUNCH_REGISTERS:
                raise RuntimeError("%s compiled at %s registers per thread: two CTAs per SM hold at most %d"
                                   % (name, r["registers"], FWD_LAUNCH_REGISTERS))
        elif ("fwd_kernel" in name or "fwd_pair_kernel" in name) and r["registers"] != FWD_LAUNCH_REGISTERS:
            raise RuntimeError("%s compiled at %s registers per thread, not %d: the setmaxnreg split of the "
                               "forward kernel would not add up" % (name, r["registers"], FWD_LAUNCH_REGISTERS))


# Kernels that must compile without register spills: the default forward (MUFU exponentials,
# every head dimension) and the backward main kernels.  The forward variants that move 6 or 8
# of every 32 exponentials to the FMA polynomial (an option, measured slower) are exempt.
NO_SPILL = (re.compile(r"fwd_kernelILi\d+ELi0ELb"), re.compile(r"bwd_main_kernel"), re.compile(r"bwd_pair_kernel"),
            re.compile(r"bwd256_kernel"), re.compile(r"fwd_pair_kernel"), re.compile(r"fwd_fp8_kernel"))


# The exception: the backward's default instance at d = 128 reads a whole dQ column (128
# values) before reducing it, so that tensor memory goes back to the MMA warp sooner; a few
# values pass through local memory.  That measured 5-7% faster on the whole backward than the
# spill-free form, so it has a budget (bytes stored and loaded) instead of zero.
# The forward's decoding configuration (two CTAs per SM) holds its softmax warpgroup at 168
# registers, below the 184 the default form's take, and keeps about 96 bytes of a score row in
# local memory.  A spill-free form (the row's maximum and exponentials in two passes over
# 32-column loads) measured about 10% slower on decoding, so that too has a budget.
SPILL_BUDGET = ((re.compile(r"bwd_main_kernelILi128ELb0E"), 192),
                (re.compile(r"fwd_kernelILi\d+ELi0ELb1E"), 160))


def check_spills(report: dict) -> None:
    for name, r in report.items():
        if not any(pat.search(name) for pat in NO_SPILL):
            continue
        budget = next((b for pat, b in SPILL_BUDGET if pat.search(name)), 0)
        if r["spill_stores"] > budget or r["spill_loads"] > budget:
            raise RuntimeError("%s spills registers (%d bytes stored, %d loaded; %d allowed)"
                               % (name, r["spill_stores"], r["spill_loads"], budget))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc] + ARCH + NVCC_FLAGS + ["-c", src, "-o", obj]
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    log = []
    failed = []
    for src, cmd, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        log.append("== %s\n%s" % (os.path.basename(src), text))
        if pr.returncode != 0:
            failed.append((src, text))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    if failed:
        msg = "\n".join("%s:\n%s" % (s, t[-4000:]) for s, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    report = ptxas_report("\n".join(log))
    check_register_split(report)
    check_spills(report)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    if verbose:
        print("\n".join(log))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
