"""Builds libmattn.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery). Translation units compile in parallel; the shared
library links the CUDA runtime statically.

build(debug=True) builds libmattn_debug.so from the same sources with
-DMATTN_DEBUG: device-side bounds checks that record and skip an access out
of range (include/mattn_debug.h), for tests."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libmattn.so")
LIB_DEBUG_PATH = os.path.join(HERE, "libmattn_debug.so")
SOURCES = ["api.cu", "mask_build.cu", "fwd_f32.cu", "fwd_tc.cu", "fwd_tc_rb.cu",
           "fwd_tc_paged.cu", "bwd_tc.cu", "bwd_tc_ragged.cu", "bwd_tc_f16.cu",
           "bwd_noalloc.cu", "varlen.cu", "combine.cu", "decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmattn.so")


def _deps() -> list:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def lib_path(debug: bool = False) -> str:
    return LIB_DEBUG_PATH if debug else LIB_PATH


def up_to_date(debug: bool = False) -> bool:
    path = lib_path(debug)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _includes(path: str) -> list:
    """Local headers a source file includes (quoted #include), resolved in
    csrc/ or include/."""
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#include \""):
                name = line.split('"')[1]
                for d in (CSRC, INCLUDE):
                    cand = os.path.join(d, name)
                    if os.path.exists(cand):
                        out.append(cand)
                        break
    return out


def _sources_of(src: str) -> set:
    """The translation unit and every local header it reaches."""
    seen, todo = set(), [os.path.join(CSRC, src)]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.add(f)
        todo.extend(_includes(f))
    return seen


def _object_stale(src: str, obj: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = _sources_of(src) | {os.path.abspath(__file__)}
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Compile every CUDA translation unit and link libmattn.so (with debug:
    libmattn_debug.so, objects apart); returns its path."""
    path = lib_path(debug)
    if not force and up_to_date(debug):
        return path
    obj_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    os.makedirs(obj_dir, exist_ok=True)
    exe = nvcc()
    flags = FLAGS + (["-DMATTN_DEBUG"] if debug else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        if not force and not ptxas_info and not _object_stale(src, obj):
            return obj
        cmd = [exe, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = path + ".tmp"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
