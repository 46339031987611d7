"""Builds libmoe.so in-tree (sparse_expert_layer_gb300/_build/) with nvcc for sm_103a.

Translation units compile in parallel; the link step makes one shared library
that exports the C ABI declared in include/moe.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoe.so")

SOURCES = ["abi.cu", "route.cu", "permute.cu", "gemv.cu", "gemm_tc.cu", "w8a8.cu", "gemv_i8.cu", "combine.cu",
           "route_noalloc.cu", "small_ffn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-I", BUILD]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe.so")
    return cand


TABLE_JSON = os.path.join(HERE, "tuning", "tile_table.json")
TABLE_INC = os.path.join(BUILD, "tile_table.inc")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe.h"))
    files.append(os.path.abspath(__file__))
    files.append(TABLE_JSON)
    return files


def write_table_inc(path: str = TABLE_INC) -> None:
    """tuning/tile_table.json -> a C table compiled into the library."""
    import json

    t = json.load(open(TABLE_JSON))
    wd = {"bf16": 0, "w8a8": 1}
    rows = [f"    {{{wd[e['wdtype']]}, {int(e['hidden'])}, {int(e['inter'])}, {int(e['bucket'])}, "
            f"{int(e['gemv_max'])}, {int(e['one_launch'])}, {int(e.get('dn_wide', 0))}}},"
            for e in t["entries"]]
    b = ", ".join(str(int(v)) for v in t["buckets"])
    text = ("// Generated from tuning/tile_table.json by build.py; do not edit.\n"
            f"static const int kTileBuckets[] = {{{b}}};\n"
            "static const TileEntry kTileTable[] = {\n" + "\n".join(rows) + "\n};\n")
    tmp = path + f".tmp{os.getpid()}"
    with open(tmp, "w") as f:
        f.write(text)
    os.replace(tmp, path)


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if stale) and return the path of libmoe.so."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest(_deps()):
        return LIB
    nvcc = _nvcc()
    objs = []
    write_table_inc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
