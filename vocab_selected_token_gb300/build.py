"""Build step for libslp.so: compiles every CUDA source under csrc/ for
sm_103a (in parallel, one process per translation unit) and links the shared
library in-tree, next to this file.  Used by ``__graft_entry__.build()``;
run directly with ``python -m vocab_selected_token_gb300.build``.

``build_checked()`` builds the bounds-checked variant, libslp_checked.so
(-DSLP_DEBUG_BOUNDS: every global access of every kernel is checked against
the buffers its call was given), in its own build folder."""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libslp.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libslp_checked.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libslp")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [__file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile and link libslp.so (or `lib`, with `extra_flags`, objects in
    `build_dir`); returns its path.  Skips the work when the library is newer
    than every source."""
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = lib + ".tmp"
    link = [cc, "-shared", *ARCH, "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        sys.stderr.write(r.stdout.decode(errors="replace"))
        raise RuntimeError(f"linking {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """The bounds-checked library (a test tool, not the product path)."""
    return build(force=force, verbose=verbose, extra_flags=("-DSLP_DEBUG_BOUNDS",),
                 lib=LIB_CHECKED, build_dir=BUILD_CHECKED)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
