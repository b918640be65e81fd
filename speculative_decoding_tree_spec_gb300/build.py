"""Build the verify library: every csrc/*.cu compiled for sm_103a in parallel, then
linked into speculative_decoding_tree_spec_gb300/_build/libspecverify.so (static
CUDA runtime, C ABI of include/spec_verify.h).  build(check=True) makes the checked
variant, _build/check/libspecverify_check.so, compiled with -DSPEC_CHECK: device-side
index checks that record what they catch in an error word (spec_check_errors)."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libspecverify.so")
CHECK_BUILD = os.path.join(BUILD, "check")
CHECK_LIB = os.path.join(CHECK_BUILD, "libspecverify_check.so")
# the files whose device code carries index checks (the other objects are shared)
CHECKED = ("api.cu", "rows.cu", "walk.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (sorted(glob.glob(os.path.join(CSRC, "*.h"))) + sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
            + [os.path.join(ROOT, "include", "spec_verify.h")])


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          check: bool = False) -> str:
    out_dir = CHECK_BUILD if check else BUILD
    lib_path = CHECK_LIB if check else LIB
    flags = NVCC_FLAGS + (["-DSPEC_CHECK"] if check else [])
    if check:
        build(force=force, verbose=verbose)  # the shared objects
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    hdrs = _headers()
    objs = []
    jobs = []
    for src in srcs:
        if check and os.path.basename(src) not in CHECKED:
            objs.append(os.path.join(BUILD, os.path.basename(src)[:-3] + ".o"))
            continue
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_info or _stale(obj, [src] + hdrs):
            cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info:
                sys.stderr.write(r.stderr)
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                check="--check" in sys.argv))
