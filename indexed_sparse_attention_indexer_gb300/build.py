"""Builds libdsi.so (and the bounds-checked libdsi_checked.so) in-tree with nvcc
for sm_103a.  Objects go to ``_build/``; the libraries sit next to this file."""
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
BUILD = os.path.join(PKG, "_build")

SOURCES = ["dsi_abi.cu", "index_score.cu", "index_score_tc.cu", "topk.cu", "sparse_mla.cu",
           "sparse_mla_tc.cu", "index_topk_prefill.cu", "dsi_static.cu",
           "mxfp8_quant.cu", "latent_fp8.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, obj: str, extra, verbose: bool):
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
           os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
    if verbose and r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def _up_to_date(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, checked: bool = True, force: bool = False) -> list:
    """Compile every source for sm_103a and link the libraries; returns their paths."""
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "dsi.h"))
    variants = [("libdsi.so", [])]
    if checked:
        variants.append(("libdsi_checked.so", ["-DDSI_CHECKED"]))
    jobs = []
    plan = []
    with cf.ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as ex:
        for lib, extra in variants:
            tag = "checked" if extra else "release"
            objs = []
            for src in SOURCES:
                obj = os.path.join(BUILD, f"{os.path.splitext(src)[0]}.{tag}.o")
                objs.append(obj)
                deps = [os.path.join(CSRC, src)] + headers
                if force or not _up_to_date(obj, deps):
                    jobs.append(ex.submit(_compile, src, obj, extra, verbose))
            plan.append((lib, objs))
        for j in jobs:
            j.result()
    out = []
    for lib, objs in plan:
        target = os.path.join(PKG, lib)
        if force or not _up_to_date(target, objs):
            cmd = [nvcc(), *ARCH, "-shared", "-o", target, *objs, "-lcudart"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed for {lib}:\n{r.stderr}")
        out.append(target)
    return out


if __name__ == "__main__":
    for p in build(verbose=True, force="--force" in sys.argv):
        print(p)
