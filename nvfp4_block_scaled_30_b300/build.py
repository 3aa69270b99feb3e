"""Build libnvfp4.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m nvfp4_block_scaled_30_b300.build [--force] [--verbose] [--checked]

Objects go to nvfp4_block_scaled_30_b300/_build/; the shared library is
written next to this file.  The CUDA runtime is linked statically and the
driver API is reached through cudaGetDriverEntryPoint, so the library loads
on machines without a GPU driver (the entry points then return
NVFP4_ERR_CUDA).
"""
import argparse
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libnvfp4.so")
# the bounds-checked variant (every access tested first; see csrc/bounds.cuh)
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libnvfp4_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
NVCC = os.environ.get("NVCC", "nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-I", INCLUDE]


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, "nvfp4.h")]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libnvfp4.so (checked=True: libnvfp4_checked.so, with
    -DNVFP4_CHECK_BOUNDS); returns the library's path."""
    bdir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    defs = ["-DNVFP4_CHECK_BOUNDS"] if checked else []
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s, *hdrs, __file__]):
            cmd = [NVCC, *ARCH, *FLAGS, *defs, "-c", s, "-o", o]
            if verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = False
    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                failed = True
                sys.stderr.write("FAILED: " + " ".join(cmd) + "\n")
    if failed:
        raise RuntimeError("nvcc failed")
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp"
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true", help="the bounds-checked variant")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, checked=a.checked))
