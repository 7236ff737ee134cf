"""Build liblp.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit is compiled for ``-gencode arch=compute_103a,code=sm_103a``
only, with ``--fmad=false`` (no multiply-add contraction: the arithmetic that
fixes the result bits is written with explicit rounding intrinsics), in
parallel, then linked into ``_build/liblp.so`` next to this file.  The build is
skipped only when ``_build/liblp.so.sha256`` records the SHA-256 of exactly the
current sources, headers, this file and the compiler flags: a library that was
copied in from elsewhere, or built from other sources, is rebuilt.  build()
prints whether it compiled.
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "liblp.so")
SOURCES = ["lp_api.cu", "lp_logits.cu", "lp_linear.cu", "lp_backward.cu"]
HEADERS = [os.path.join(ROOT, "include", "lp.h")] + [
    os.path.join(CSRC, f) for f in ("lp_device.cuh", "lp_internal.h", "lp_tcgen05.cuh",
                                    "lp_check.cuh")
]
# the checked build (-DLP_CHECKED: index and coordinate tests in every kernel)
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "liblp.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "--fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblp")
    return path


def _paths(checked: bool):
    return (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)


def source_hash(checked: bool = False) -> str:
    """SHA-256 over the sources, headers, this build script and the flags."""
    h = hashlib.sha256()
    if checked:
        h.update(b"LP_CHECKED")
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    for path in deps:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def _stale(checked: bool = False) -> bool:
    _, lib = _paths(checked)
    stamp = lib + ".sha256"
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return True
    with open(stamp) as f:
        return f.read().strip() != source_hash(checked)


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = False,
          checked: bool = False) -> str:
    """Compile liblp.so unless it was built from exactly these sources; return its path.
    checked=True builds the checked library (_build_checked/liblp.so) instead."""
    build_dir, lib = _paths(checked)
    what = "checked liblp" if checked else "liblp"
    if not force and not _stale(checked):
        if not quiet:
            print(f"{what}: up to date (sources sha256 {source_hash(checked)[:16]})", flush=True)
        return lib
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checked:
        extra += ["-DLP_CHECKED"]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    digest = source_hash(checked)
    with open(lib + ".sha256", "w") as f:
        f.write(digest + "\n")
    if not quiet:
        print(f"{what}: compiled {len(SOURCES)} sources for sm_103a (sources sha256 {digest[:16]})",
              flush=True)
    return lib


if __name__ == "__main__":
    print(build(force=True))
