"""Build libgemm_f32.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then the objects are linked into
dense_fp32_gemm_major_gb300/libgemm_f32.so (CUDA runtime linked statically,
no libcuda link: the driver's tensor-map encoder is looked up at run time, so
the library also loads on machines without a GPU driver).

The checked build, libgemm_f32_checked.so, is the same sources compiled with
GEMM_F32_INDEX_CHECKS=1 (device-side index checks, csrc/checks.cuh) into
_build/checked/; build_all() compiles both libraries' units in one pool.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgemm_f32.so")
OBJ_DIR_CHECKED = os.path.join(OBJ_DIR, "checked")
LIB_CHECKED = os.path.join(PKG, "libgemm_f32_checked.so")
CHECKED_FLAGS = ["-DGEMM_F32_INDEX_CHECKS=1"]
SOURCES = ["api.cu", "simt_gemm.cu", "tc_gemm.cu", "transpose.cu", "pack.cu", "reduce.cu",
           "probe.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xcompiler", "-Wall", "-Wno-deprecated-gpu-targets"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _deps():
    return (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
            + [os.path.abspath(__file__)])


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra, obj_dir: str = OBJ_DIR) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj


def _link(objs, lib: str, verbose: bool) -> str:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}")
    return lib


def _variants(checked_too: bool):
    out = [(LIB, OBJ_DIR, [])]
    if checked_too:
        out.append((LIB_CHECKED, OBJ_DIR_CHECKED, CHECKED_FLAGS))
    return out


def _build(variants, force: bool, extra_flags, verbose: bool):
    deps = _deps()
    todo = [v for v in variants if force or extra_flags or _stale(v[0], deps)]
    if not todo:
        return
    for _, obj_dir, _ in todo:
        os.makedirs(obj_dir, exist_ok=True)
    jobs = [(src, list(flags) + list(extra_flags), obj_dir)
            for _, obj_dir, flags in todo for src in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(*j), jobs))
    for i, (lib, _, _) in enumerate(todo):
        _link(objs[i * len(SOURCES):(i + 1) * len(SOURCES)], lib, verbose)


def build_library(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libgemm_f32.so."""
    _build(_variants(False), force, extra_flags, verbose)
    return LIB


def build_all(force: bool = False, verbose: bool = False):
    """Compile (if stale) libgemm_f32.so and libgemm_f32_checked.so together;
    return both paths."""
    _build(_variants(True), force, (), verbose)
    return LIB, LIB_CHECKED


if __name__ == "__main__":
    build_all(force=True, verbose=True)
