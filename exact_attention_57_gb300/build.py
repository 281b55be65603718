"""Build the sm_103a shared library ``libfa.so`` in-tree with nvcc.

Each translation unit under ``csrc/`` is compiled in parallel to an object
file, then linked into ``exact_attention_57_gb300/libfa.so``.  ptxas
statistics (registers, spills, shared memory) are kept in
``exact_attention_57_gb300/_build/ptxas.log``.

``build_library(debug=True)`` builds ``libfa_debug.so`` (objects in
``_build_debug/``) with ``-DFA_DEBUG``: the kernels then check the index of
every plain global load and store and report a failed check in the status
word (bit 32) instead of making the access.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libfa_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden",
              "-Xptxas", "-v", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DFA_DEBUG"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    headers = (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
               + glob.glob(os.path.join(INCLUDE, "*.h")))
    srcs = sources()
    objs, procs = [], []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc(), *ARCH, *flags, "-c", src, "-o", obj]
            log = open(obj + ".log", "w")
            procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, pr, log in procs:
        pr.wait()
        log.close()
        if pr.returncode != 0:
            failed.append(src)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as out:
        for obj in objs:
            if os.path.exists(obj + ".log"):
                out.write(open(obj + ".log").read())
    if failed:
        msgs = "".join(open(os.path.join(build_dir, os.path.basename(s)[:-3] + ".o.log")).read()
                       for s in failed)
        raise RuntimeError(f"nvcc failed for {failed}:\n{msgs[-6000:]}")
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(build_dir, "ptxas.log")).read())
    return lib


def ptxas_summary(log_path: str | None = None) -> str:
    """Markdown table of the ptxas statistics of every kernel in the last
    build: registers per thread, stack frame, spill stores and loads, static
    shared memory (the tensor-core kernels' shared memory is dynamic and set
    at launch).  Kernel names are demangled with c++filt when it is present."""
    import re
    text = open(log_path or os.path.join(BUILD, "ptxas.log")).read()
    rows, cur = [], None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = {"name": m.group(1), "regs": "?", "stack": "?", "spill_st": "?",
                   "spill_ld": "?", "smem": "0"}
            rows.append(cur)
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                      line)
        if m:
            cur["stack"], cur["spill_st"], cur["spill_ld"] = m.groups()
        m = re.search(r"Used (\d+) registers", line)
        if m:
            cur["regs"] = m.group(1)
        m = re.search(r"(\d+) bytes smem", line)
        if m:
            cur["smem"] = m.group(1)
    names = [r["name"] for r in rows]
    filt = shutil.which("c++filt")
    if filt and names:
        out = subprocess.run([filt], input="\n".join(names), capture_output=True, text=True)
        dem = out.stdout.splitlines()
        if len(dem) == len(names):
            for r, n in zip(rows, dem):
                n = n.replace("(anonymous namespace)::", "")
                r["name"] = re.sub(r"\([^()]*\)$", "", n)
    lines = ["| kernel | registers | stack (B) | spill stores (B) | spill loads (B) | static smem (B) |",
             "|---|---|---|---|---|---|"]
    for r in sorted(rows, key=lambda r: r["name"]):
        lines.append(f"| `{r['name']}` | {r['regs']} | {r['stack']} | {r['spill_st']} | "
                     f"{r['spill_ld']} | {r['smem']} |")
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    if "--ptxas-summary" in sys.argv:
        build_library(force="--force" in sys.argv)
        print(ptxas_summary(), end="")
    else:
        print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
