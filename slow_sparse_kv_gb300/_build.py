"""In-tree build of libsfi (and of the workload generator) for sm_103a.

Each translation unit is compiled by nvcc in parallel; the objects are linked
into ``_lib/libsfi.so`` with the CUDA runtime linked statically.  A unit is
rebuilt only when a source or header is newer than its object.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, obj: str, deps, include_dirs, verbose: bool) -> str:
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest(deps + [src, __file__]):
        return obj
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *[f"-I{d}" for d in include_dirs], "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr.strip():
        print(r.stderr, flush=True)
    return obj


def build_library(src_dir: str, out_dir: str, name: str, include_dirs, verbose=False,
                  jobs: int | None = None) -> str:
    os.makedirs(os.path.join(out_dir, "obj"), exist_ok=True)
    srcs = sorted(os.path.join(src_dir, f) for f in os.listdir(src_dir)
                  if f.endswith((".cu", ".cpp")))
    deps = [os.path.join(src_dir, f) for f in os.listdir(src_dir) if f.endswith((".h", ".cuh"))]
    for d in include_dirs:
        deps += [os.path.join(d, f) for f in os.listdir(d) if f.endswith(".h")]
    objs = [os.path.join(out_dir, "obj", os.path.basename(s) + ".o") for s in srcs]
    jobs = jobs or max(1, min(len(srcs), os.cpu_count() or 4))
    with ThreadPoolExecutor(jobs) as ex:
        list(ex.map(lambda so: _compile(so[0], so[1], deps, include_dirs, verbose), zip(srcs, objs)))
    lib = os.path.join(out_dir, name)
    if not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        cmd = [nvcc(), *ARCH, "-shared", "-o", lib + ".tmp", *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {name} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(lib + ".tmp", lib)
    return lib


def build(verbose: bool = False) -> list:
    """Build libsfi and the workload generator library; return their paths."""
    pkg = os.path.dirname(os.path.abspath(__file__))
    out = [build_library(os.path.join(pkg, "csrc"), os.path.join(pkg, "_lib"), "libsfi.so",
                         [os.path.join(ROOT, "include")], verbose)]
    gen = os.path.join(ROOT, "sfi_workloads")
    out.append(build_library(os.path.join(gen, "csrc"), os.path.join(gen, "_lib"), "libsfigen.so",
                             [os.path.join(ROOT, "include")], verbose))
    return out


if __name__ == "__main__":
    for p in build(verbose=True):
        print(p)
