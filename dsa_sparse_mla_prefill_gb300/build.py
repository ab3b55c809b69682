"""Builds the sm_103a libraries in-tree (no cmake, no torch extension).

    python -m dsa_sparse_mla_prefill_gb300.build [--verbose]

Produces, next to this file:
  libdsa.so           the C-ABI library declared in include/dsa.h
  libdsa_selftest.so  a tcgen05 layout self-test used only by the tests
Each .cu is compiled in parallel with
  nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3 -Xptxas -v
and the ptxas resource report is kept in _build/ptxas.log.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_SOURCES = ["dsa_api.cu", "sparse_prefill.cu", "union_build.cu", "key_mask.cu", "grouped_prefill.cu",
               "masked_mha.cu", "index_convert.cu", "dispatch.cu", "host_pipeline.cu", "host_noalloc.cu",
               "wait_probe.cu", "kv_fp8.cu"]
SELFTEST_SOURCES = ["selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-use_fast_math", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the sm_103a libraries need the CUDA 13 toolkit")


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _up_to_date(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, s) for s in sources] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                                       if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "dsa.h"))
    deps.append(os.path.abspath(__file__))
    return all(os.path.getmtime(d) <= t for d in deps if os.path.exists(d))


def build(verbose: bool = False, force: bool = False) -> dict:
    os.makedirs(BUILD, exist_ok=True)
    targets = {
        os.path.join(HERE, "libdsa.so"): LIB_SOURCES,
        os.path.join(HERE, "libdsa_selftest.so"): SELFTEST_SOURCES,
    }
    todo = {t: s for t, s in targets.items() if force or not _up_to_date(t, s)}
    if not todo:
        return {t: "up to date" for t in targets}
    srcs = sorted({s for ss in todo.values() for s in ss})
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = dict(zip(srcs, ex.map(_compile, srcs)))
    for s in srcs:
        logs.append(f"==== {s}\n{results[s][1]}")
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    for target, ss in todo.items():
        objs = [results[s][0] for s in ss]
        tmp = target + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed for {target}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, target)
    if verbose:
        print("\n".join(logs))
    return {t: ("built" if t in todo else "up to date") for t in targets}


if __name__ == "__main__":
    res = build(verbose="--verbose" in sys.argv, force="--force" in sys.argv)
    for k, v in res.items():
        print(f"{os.path.basename(k)}: {v}")
