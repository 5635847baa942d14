"""Build libiha.so (the CUDA library behind include/iha.h) in-tree for sm_103a.

Each translation unit under csrc/ is compiled in parallel with nvcc, then linked
into transformer_attention_variant_gb300/libiha.so.  Object files go to _build/
at the repository root.  Re-running only recompiles what changed.

Warp-specialised kernels that move registers between their warpgroups with
setmaxnreg are only correct when compiled to exactly the per-thread register
count their split assumes (a warpgroup that asks for more registers than the
launch provided waits forever).  ptxas reports each kernel's count; the build
fails when a kernel listed in REG_CONTRACTS does not match the constant its
source declares.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libiha.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


# kernel-name fragment -> (source file, constant holding the launch register count)
REG_CONTRACTS = {
    "attn_fwd_tc": ("k_attention_tc.cu", "AT_LAUNCH_REGS"),
    "bwd_attn_tc": ("k_backward_tc.cu", "BA_LAUNCH_REGS"),
    "proj_mix_tc": ("k_project_mix_tc.cu", "PM_LAUNCH_REGS"),
}


def _declared_regs(src: str, const: str) -> int:
    with open(os.path.join(CSRC, src)) as f:
        m = re.search(r"\b" + const + r"\s*=\s*(\d+)", f.read())
    if not m:
        raise RuntimeError(f"{src}: constant {const} not found")
    return int(m.group(1))


def _kernel_registers(log: str) -> dict:
    """Mangled kernel name -> registers per thread, from ptxas -v output."""
    regs, cur = {}, None
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            regs[cur] = int(m.group(1))
            cur = None
    return regs


def check_register_contracts() -> None:
    """Fail unless every kernel named in REG_CONTRACTS was compiled to its declared count."""
    problems = []
    for frag, (src, const) in REG_CONTRACTS.items():
        log_path = os.path.join(BUILD, src[:-3] + ".ptxas.txt")
        if not os.path.exists(log_path):
            problems.append(f"{src}: no ptxas report (rebuild with force=True)")
            continue
        with open(log_path) as f:
            regs = _kernel_registers(f.read())
        want = _declared_regs(src, const)
        found = {k: v for k, v in regs.items() if frag in k}
        if not found:
            problems.append(f"{src}: no kernel named like {frag} in the ptxas report")
        for k, v in found.items():
            if v != want:
                problems.append(f"{k}: {v} registers per thread, its register split needs {const} = {want}")
    if problems:
        raise RuntimeError("register contract violated:\n  " + "\n  ".join(problems))


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _mtime(p):
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    hdr_time = max(_mtime(h) for h in _headers())
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        log = obj[:-2] + ".ptxas.txt"
        if force or ptxas_verbose or _mtime(obj) < max(_mtime(src), hdr_time) or not os.path.exists(log):
            jobs.append(([nvcc, "-Xptxas=-v", *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj], log))

    def run(job):
        cmd, log = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            with open(log, "w") as f:
                f.write(r.stdout + r.stderr)
        return cmd, r

    failed = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if ptxas_verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                elif verbose:
                    sys.stderr.write(" ".join(cmd[-3:]) + "\n")
                if r.returncode != 0:
                    failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    check_register_contracts()
    if force or jobs or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libiha.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv)
    print(LIB)
