"""Build libpagedkv.so in-tree for sm_103a with nvcc.

``python -m paged_kv_cache_70_gb300.build`` (or ``build()``) compiles every
``csrc/*.cu`` translation unit in parallel and links them into
``_build/libpagedkv.so`` next to this file.  ``decode.cu``, ``write.cu`` and
``prefill.cu`` are not units of their own: ``step.cu`` includes them, so that
its one-launch step kernel can run their CTA functions.  The CUDA runtime is
linked statically, so the library needs only the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")
    return cand


# sources compiled inside step.cu
INCLUDED = ("decode.cu", "write.cu", "prefill.cu")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu") and f not in INCLUDED)


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra: tuple[str, ...] = ()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
               if f.endswith((".cuh", ".h")) or f in INCLUDED]
    headers.append(os.path.join(INCLUDE, "pagedkv.h"))
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
            jobs.append(cmd)
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True),
                                  jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libpagedkv.so failed")
        os.replace(tmp, LIB)
    return LIB


def build_variant(tag: str, defines: tuple[str, ...], variant_sources: tuple[str, ...]) -> str:
    """A library built with extra `defines` in the translation units named in
    `variant_sources` (file names under csrc/) and the default objects for the
    rest, at _build/<tag>/libpagedkv.so.  Used by tests that need a kernel
    compiled differently (e.g. a shorter wait limit); the default library is
    untouched."""
    build()
    out_dir = os.path.join(BUILD, tag)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    for src in sources():
        name = os.path.basename(src)
        if name in variant_sources:
            obj = os.path.join(out_dir, name[:-3] + ".o")
            cmd = [nvcc, *ARCH, *FLAGS, *defines, "-I", INCLUDE, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
        else:
            obj = os.path.join(BUILD, name[:-3] + ".o")
        objs.append(obj)
    lib = os.path.join(out_dir, "libpagedkv.so")
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", lib, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"link of {lib} failed")
    return lib


if __name__ == "__main__":
    defines = tuple(a for a in sys.argv[1:] if a.startswith("-D"))
    print(build(force="--force" in sys.argv or bool(defines), verbose="-v" in sys.argv,
                extra=defines))
