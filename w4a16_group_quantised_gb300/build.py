"""Build libw4a16.so from csrc/ with nvcc for sm_103a (in-tree, no cmake).

Each translation unit compiles in parallel; the objects link into one shared
library next to this file.  Rebuilds only when a source is newer than the
library.

variant="trace" builds libw4a16_trace.so instead: the same sources with
W4A16_DECODE_TRACE defined, which compiles the decode kernel's per-CTA
timeline stamps in (a profiling build; the default library has none of
them).  The binding loads it when W4A16_LIBRARY=trace.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "libw4a16.so")
BUILD_DIR = os.path.join(HERE, "_build")
VARIANTS = {None: (OUT, BUILD_DIR, []),
            "trace": (os.path.join(HERE, "libw4a16_trace.so"), os.path.join(HERE, "_build_trace"),
                      ["-DW4A16_DECODE_TRACE=1"])}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "w4a16.h"), __file__]


def _variant(variant):
    if variant not in VARIANTS:
        raise ValueError(f"unknown build variant {variant!r}; known: None, 'trace'")
    return VARIANTS[variant]


def up_to_date(variant=None) -> bool:
    out = _variant(variant)[0]
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None, variant=None) -> str:
    out, build_dir, vflags = _variant(variant)
    if not force and up_to_date(variant):
        return out
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = NVCC_FLAGS + vflags + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(_sources()))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                variant="trace" if "--trace" in sys.argv else None))
