"""Build ``libep_gb300.so`` (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel to an object file
under ``_build/``, then linked into ``combine_router_softmax_gb300/libep_gb300.so``
(CUDA runtime linked statically). ptxas resource usage (``-Xptxas -v``) goes
to ``_build/ptxas.log``.

Run ``python combine_router_softmax_gb300/build.py`` or call :func:`build`. This file
is self-contained (it never imports the package, whose import loads the
library), so other scripts load it by file path before the library exists.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import pathlib
import shutil
import subprocess
import sys

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = ROOT / "_build"
LIB = PKG / "libep_gb300.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              f"-I{ROOT / 'include'}", "--expt-relaxed-constexpr"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and pathlib.Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def sources() -> list[pathlib.Path]:
    return sorted(CSRC.glob("*.cu"))


def _inputs_mtime() -> float:
    files = list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")) + list((ROOT / "include").glob("*.h"))
    files.append(pathlib.Path(__file__))
    return max(f.stat().st_mtime for f in files)


def _compile(nvcc: str, src: pathlib.Path) -> tuple[pathlib.Path, str]:
    obj = BUILD / (src.stem + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", str(src), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> pathlib.Path:
    """Compile and link the library if any source is newer than it."""
    if not force and LIB.exists() and LIB.stat().st_mtime >= _inputs_mtime():
        return LIB
    nvcc = nvcc_path()
    BUILD.mkdir(exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s), srcs))
    log = "\n".join(f"== {o.name}\n{msg}" for o, msg in results)
    (BUILD / "ptxas.log").write_text(log)
    if verbose:
        print(log)
    tmp = LIB.with_name(LIB.name + f".tmp{os.getpid()}")
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *[str(o) for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
