"""Builds the package's native parts in-tree, into ``_lib/``.

* ``libpagedkv.so`` -- the CUDA library behind ``include/pagedkv.h``, compiled
  for sm_103a only (``-gencode arch=compute_103a,code=sm_103a``); the
  translation units compile in parallel and link with the static CUDA runtime.
* ``libpkvgen.so`` -- the seeded input generator (plain C, no CUDA).

Nothing here runs at import time: ``paged_kv_cache_11_gb300`` loads the
libraries and fails loudly when they have not been built.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
LIBDIR = PKG / "_lib"
CUDA_SOURCES = ["api.cu", "decode.cu", "group_prefix.cu", "append_copy.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(home) / "bin" / "nvcc"
    if cand.exists():
        return str(cand)
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def _stale(target: Path, deps: list[Path]) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(d.stat().st_mtime > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> Path:
    LIBDIR.mkdir(exist_ok=True)
    out = LIBDIR / "libpagedkv.so"
    deps = [CSRC / s for s in CUDA_SOURCES] + [CSRC / "pkv_internal.cuh", CSRC / "decode_common.cuh",
                                                PKG.parent / "include" / "pagedkv.h"]
    if not force and not _stale(out, deps):
        return out
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    objs = [LIBDIR / (Path(s).stem + ".o") for s in CUDA_SOURCES]
    with ThreadPoolExecutor(len(CUDA_SOURCES)) as ex:
        list(ex.map(lambda so: _run([nvcc, *flags, "-c", str(CSRC / so[0]), "-o", str(so[1])]),
                    zip(CUDA_SOURCES, objs)))
    tmp = out.with_suffix(".so.tmp")
    _run([nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)])
    os.replace(tmp, out)
    return out


def build_generator(force: bool = False) -> Path:
    LIBDIR.mkdir(exist_ok=True)
    src = PKG / "gen" / "pkv_gen.c"
    out = LIBDIR / "libpkvgen.so"
    if not force and not _stale(out, [src]):
        return out
    tmp = out.with_suffix(".so.tmp")
    _run(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread", str(src), "-o", str(tmp), "-lm"])
    os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> None:
    build_generator(force)
    build_library(force)


if __name__ == "__main__":
    build_all(force=True)
