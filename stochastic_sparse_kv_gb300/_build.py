"""In-tree build of libsanta.so for sm_103a (nvcc, no cmake; translation units compiled
in parallel).  Run as a module or call build()."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsanta.so")
UNITS = ["santa_api.cu", "santa_kernels_d128.cu", "santa_kernels_d64.cu"]
HEADERS = ["santa_common.cuh", "santa_sample.cuh", "santa_tcgen05.cuh", "santa_score.cuh", "santa_gather.cuh", "santa_dense.cuh",
           "santa_cluster.cuh", "santa_kernels.h"]
# the timeline build: the same sources with %globaltimer stamps (santa_timeline_buffer)
TIMELINE_LIB = os.path.join(HERE, "libsanta_timeline.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsanta.so")
    return p


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, timeline: bool = False) -> str:
    """Build libsanta.so (timeline=True: libsanta_timeline.so, compiled with -DSANTA_TIMELINE
    into its own object folder); returns the library's path."""
    out_dir, lib, extra = (OUT_DIR + "_timeline", TIMELINE_LIB, ["-DSANTA_TIMELINE"]) if timeline else (OUT_DIR, LIB, [])
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "santa.h")]
    objs, jobs = [], []
    for u in UNITS:
        src = os.path.join(CSRC, u)
        obj = os.path.join(out_dir, u.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            if ptxas_v:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_v or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv, timeline="--timeline" in sys.argv))
