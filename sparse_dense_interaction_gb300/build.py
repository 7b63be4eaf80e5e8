"""In-tree build of the CUDA libraries (sm_103a only).

* ``_build/libdlrm_sparse.so``   -- the DLRM sparse path's C ABI
  (``include/dlrm_sparse.h``), from ``csrc/*.cu``;
* ``_build/libdlrm_workloads.so`` -- device-side input generation for the
  synthetic workloads, from ``workloads_csrc/*.cu``.

Translation units compile in parallel with nvcc, one ``-gencode``
(``arch=compute_103a,code=sm_103a``), then link as shared libraries with the
static CUDA runtime.  A library is rebuilt only when a source or header is
newer than it.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
NVCC_FLAGS = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "--expt-relaxed-constexpr", "-I", INCLUDE]

LIBS = {
    "libdlrm_sparse.so": os.path.join(HERE, "csrc"),
    "libdlrm_workloads.so": os.path.join(HERE, "workloads_csrc"),
}


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources(src_dir):
    return sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith(".cu"))


def _deps(src_dir):
    files = [os.path.join(src_dir, f) for f in os.listdir(src_dir)
             if f.endswith((".cu", ".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def lib_path(name: str) -> str:
    return os.path.join(BUILD, name)


def _up_to_date(target, deps):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _compile(src, obj, extra):
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> dict:
    """Builds both libraries; returns {name: path}."""
    os.makedirs(BUILD, exist_ok=True)
    out = {}
    for name, src_dir in LIBS.items():
        target = lib_path(name)
        out[name] = target
        if not force and not extra_flags and _up_to_date(target, _deps(src_dir)):
            continue
        objdir = os.path.join(BUILD, name.replace(".so", "_obj"))
        os.makedirs(objdir, exist_ok=True)
        srcs = _sources(src_dir)
        objs = [os.path.join(objdir, os.path.basename(s).replace(".cu", ".o")) for s in srcs]
        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
            logs = list(ex.map(lambda so: _compile(so[0], so[1], list(extra_flags)), zip(srcs, objs)))
        if verbose:
            for s, log in zip(srcs, logs):
                if log.strip():
                    print(f"--- {os.path.basename(s)}\n{log}")
        tmp = target + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp] + objs, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {name} failed:\n{r.stderr}")
        os.replace(tmp, target)
    return out


if __name__ == "__main__":
    import sys
    extra = ["-Xptxas", "-v"] if "-v" in sys.argv else []
    for k, v in build(force="-f" in sys.argv or bool(extra), verbose=True, extra_flags=extra).items():
        print(k, v)
