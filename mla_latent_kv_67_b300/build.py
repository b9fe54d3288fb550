"""Build ``libmla_b300.so`` from ``csrc/`` with nvcc for sm_103a, in-tree.

``python -m mla_latent_kv_67_b300.build [--ptxas-v]``
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libmla_b300.so")
# The same sources compiled with MLA_TEST_HOOKS: shortened device wait
# limits and mla_test_withhold_pages (include/mla_b300_test.h), for the
# tests that make a bounded wait run out. Never the shipped library.
HOOK_LIB = os.path.join(LIBDIR, "libmla_b300_testhooks.so")
OBJDIR = os.path.join(os.path.dirname(HERE), "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _newest_header() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(os.path.dirname(HERE), "include", "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(ptxas_verbose: bool = False, force: bool = False, quiet: bool = True,
          hooks: bool = False) -> str:
    lib = HOOK_LIB if hooks else LIB
    objdir = os.path.join(OBJDIR, "hooks") if hooks else OBJDIR
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _newest_header()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "--expt-relaxed-constexpr", "-I", os.path.dirname(HERE)]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    if hooks:
        flags += ["-DMLA_TEST_HOOKS"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        if (not force and not ptxas_verbose and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_t)):
            return obj, ""
        cmd = [nvcc(), "-c", src, "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    logs = "".join(l for _, l in results)
    if logs and (ptxas_verbose or not quiet):
        sys.stderr.write(logs)
    objs = [o for o, _ in results]
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "shared",
                                                              "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(ptxas_verbose="--ptxas-v" in sys.argv, force="--force" in sys.argv, quiet=False,
                hooks="--hooks" in sys.argv))
