"""Builds libpagedkv.so in-tree (paged_kv_gqa_03_gb300/_build/) with nvcc for
sm_103a.  Translation units compile in parallel; a unit is rebuilt only when
it or a header changed.

    python paged_kv_gqa_03_gb300/build.py [--force] [--ptxas-info]
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile(src, obj, ptxas_info):
    cmd = [_nvcc()] + FLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    newest_header = max(os.path.getmtime(h) for h in _headers())
    jobs = []
    for src in sources:
        obj = os.path.join(OUT, os.path.basename(src) + ".o")
        stale = (force or ptxas_info or not os.path.exists(obj)
                 or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header))
        jobs.append((src, obj, stale))
    todo = [(s, o) for s, o, st in jobs if st]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4)) as ex:
            futs = {ex.submit(_compile, s, o, ptxas_info): s for s, o in todo}
            for f in cf.as_completed(futs):
                log = f.result()
                if (verbose or ptxas_info) and log:
                    print(f"== {os.path.basename(futs[f])}\n{log}", file=sys.stderr)
    objs = [o for _, o, _ in jobs]
    if todo or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_info="--ptxas-info" in sys.argv, verbose=True))
