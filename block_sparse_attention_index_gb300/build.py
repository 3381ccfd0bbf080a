"""Build the MSA CUDA library for sm_103a, in-tree.

Each translation unit under csrc/ is compiled by nvcc in parallel, then the
objects are linked into block_sparse_attention_index_gb300/_lib/libmsa_gb300.so
(CUDA runtime linked statically).  Rebuilds only what changed, and everything
when the objects were made on another machine, by another nvcc or with other
flags (a stamp file records those).  Prints one line saying what it did.
"""
from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libmsa_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                "-I", CSRC, "-I", INCLUDE]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers_mtime():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src, hdr_mtime, extra, verbose):
    obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_mtime):
        return obj, ""
    cmd = [NVCC] + FLAGS + extra + ["-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return obj, (res.stdout + res.stderr) if verbose else ""


def _stamp() -> str:
    ver = subprocess.run([NVCC, "--version"], capture_output=True, text=True).stdout.strip().splitlines()
    return "\n".join([platform.machine(), ver[-1] if ver else "nvcc ?", " ".join(FLAGS)]) + "\n"


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    stamp, stamp_file = _stamp(), os.path.join(OBJ_DIR, "stamp.txt")
    try:
        same = open(stamp_file).read() == stamp
    except OSError:
        same = False
    if not same:  # objects (if any) from another machine, compiler or flag set: start over
        for d in (OBJ_DIR, LIB_DIR):
            shutil.rmtree(d, ignore_errors=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    hdr = _headers_mtime()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    srcs = _sources()
    stale = [s for s in srcs if not os.path.exists(os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o")) or
             os.path.getmtime(os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o")) <
             max(os.path.getmtime(s), hdr)]
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, hdr, extra, verbose or ptxas_info), srcs))
    objs = [o for o, _ in results]
    for _, log in results:
        if log:
            print(log)
    linked = False
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
        linked = True
    with open(stamp_file, "w") as f:
        f.write(stamp)
    mode = "full" if not same else ("incremental" if stale else "up to date")
    print(f"msa build ({platform.machine()}, sm_103a): {mode}; compiled {len(stale)} of {len(srcs)} translation "
          f"units; library {'linked' if linked else 'unchanged'}: {LIB}")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
